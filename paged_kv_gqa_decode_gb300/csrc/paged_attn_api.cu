// C ABI of the paged-KV GQA decode library (include/paged_attn.h): argument
// validation, launch planning (grid, pipeline depth, workspace), TMA tensor
// maps, and the per-device workspace the plain entry point owns.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "append.h"
#include "launch.h"
#include "paged_attn.h"

namespace pagedattn {
namespace {

thread_local int g_last_cuda_error = 0;
thread_local int g_launch_flags = 0;  // paged_attn_set_launch_flags

constexpr int kMaxSeqsPerLaunch = 4096;
constexpr size_t kWsAlign = 256;
constexpr int kAppendApartPieces = 4;  // (s, g) pieces per CTA from which the append runs apart
constexpr int kMaxMultiRows = 256;      // multi-token decode: max q_len * G (16 pieces of 16 rows)
constexpr long long kRingBytesPerSm = 128 << 10;            // K/V rings of one SM, few pieces per CTA
constexpr long long kRingBytesPerSmManyPieces = 160 << 10;  // ... two or more pieces per CTA

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int cuda_fail(int err) {
  g_last_cuda_error = err;
  return PAGED_ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int validate_sizes(int num_seqs, int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                   int block_size) {
  if (H_kv <= 0 || H_q <= 0 || H_q % H_kv != 0 || H_q / H_kv > 16) return PAGED_ATTN_ERR_HEADS;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PAGED_ATTN_ERR_HEAD_DIM;
  if (block_size != 16 && block_size != 32) return PAGED_ATTN_ERR_BLOCK_SIZE;
  if (num_seqs < 0 || max_blocks_per_seq <= 0) return PAGED_ATTN_ERR_SIZES;
  // lengths up to max_blocks_per_seq * block_size must fit int32; table rows must be indexable
  if ((long long)max_blocks_per_seq * block_size > 0x7fffffffLL) return PAGED_ATTN_ERR_SIZES;
  if ((long long)H_kv * block_size > 0x7fffffffLL) return PAGED_ATTN_ERR_SIZES;
  return PAGED_ATTN_OK;
}

struct DeviceInfo {
  int sms = 0;
  int max_smem = 0;     // opt-in dynamic shared memory per block
  int smem_per_sm = 0;  // shared memory per multiprocessor
};

struct OwnedWorkspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};

// Per-device state, indexed by device ordinal (guarded by g_mu).
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
OwnedWorkspace g_ws[kMaxDevices];
void* g_static_scratch_ptr[kMaxDevices];  // address of the static scratch array

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (*dev < 0 || *dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  return PAGED_ATTN_OK;
}

int device_info(DeviceInfo* out) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != PAGED_ATTN_OK) return rc;
  cudaError_t e;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_info[dev].sms > 0) {
    *out = g_info[dev];
    return PAGED_ATTN_OK;
  }
  DeviceInfo di;
  if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&di.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                  dev)) != cudaSuccess)
    return cuda_fail(e);
  g_info[dev] = di;
  *out = di;
  return PAGED_ATTN_OK;
}

// Everything a launch needs that depends only on sizes and the device.
struct Plan {
  int D, BS, G;
  bool g16;
  bool fp8;     // FP8 caches
  bool xp;      // x-packed K / D-major V caches (bf16)
  int rows;     // query rows of one piece: G, or a multi-token chunk (8 or 16)
  int qchunks;  // multi-token decode: pieces per (sequence, KV head); 0: single token
  int chunk;    // sequences per launch
  int stages;   // pipeline depth
  size_t smem;  // dynamic shared memory per CTA
  int grid;     // persistent CTAs
  size_t off_counters, off_partials, ws_bytes;
};

// G: query rows of one piece; qchunks > 0: multi-token decode (room for chunk + 1
// row offsets and the page prefixes of qchunks passes).
template <int D, int BS, bool FP8>
bool plan_smem(int G, int chunk, int max_smem, long long ring_cap, int qchunks, int* stages,
               size_t* smem) {
  using L = SmemLayout<D, BS, FP8>;
  const int qo_entries = qchunks > 0 ? chunk + 1 : 0;
  const int walks = qchunks > 0 ? qchunks : 1;
  const L none{0, G, chunk, qo_entries, walks};
  const long long fixed = none.total() + 2048;  // + alignment slack and static shared memory
  const long long per_stage = L::kStageBytes + L::kScaleBytes + 16;
  long long st = (max_smem - fixed) / per_stage;
  if (st > kMaxStages) st = kMaxStages;
  if (st > ring_cap / L::kStageBytes) st = ring_cap / L::kStageBytes;
  // At least one slot per consumer warp (slot s belongs to warp s % 4).
  if (st < kConsumerWarps) return false;
  const L lay{(int)st, G, chunk, qo_entries, walks};
  *stages = (int)st;
  *smem = (size_t)lay.total() + 1024;
  return *smem + 256 <= (size_t)max_smem;  // + the kernel's static shared memory
}

template <bool FP8>
bool plan_smem_d(int D, int BS, int G, int chunk, int max_smem, long long ring_cap,
                 int qchunks, int* stages, size_t* smem) {
  if (D == 64) {
    if constexpr (FP8) return false;  // FP8 caches need head_dim 128 or 256
    else
      return BS == 16 ? plan_smem<64, 16, false>(G, chunk, max_smem, ring_cap, qchunks, stages, smem)
                      : plan_smem<64, 32, false>(G, chunk, max_smem, ring_cap, qchunks, stages, smem);
  }
  if (D == 128)
    return BS == 16 ? plan_smem<128, 16, FP8>(G, chunk, max_smem, ring_cap, qchunks, stages, smem)
                    : plan_smem<128, 32, FP8>(G, chunk, max_smem, ring_cap, qchunks, stages, smem);
  return BS == 16 ? plan_smem<256, 16, FP8>(G, chunk, max_smem, ring_cap, qchunks, stages, smem)
                  : plan_smem<256, 32, FP8>(G, chunk, max_smem, ring_cap, qchunks, stages, smem);
}

bool plan_smem_any(int D, int BS, bool fp8, int G, int chunk, int max_smem, long long ring_cap,
                   int qchunks, int* stages, size_t* smem) {
  return fp8 ? plan_smem_d<true>(D, BS, G, chunk, max_smem, ring_cap, qchunks, stages, smem)
             : plan_smem_d<false>(D, BS, G, chunk, max_smem, ring_cap, qchunks, stages, smem);
}

// rows > 0: multi-token decode with `rows` query rows per piece and `qchunks`
// pieces per (sequence, KV head).
int make_plan(int num_seqs, int H_q, int H_kv, int D, int BS, const DeviceInfo& di, Plan* pl,
              bool fp8 = false, int rows = 0, int qchunks = 0) {
  pl->D = D;
  pl->fp8 = fp8;
  pl->xp = false;
  pl->BS = BS;
  pl->G = H_q / H_kv;
  pl->rows = rows > 0 ? rows : pl->G;
  pl->qchunks = rows > 0 ? qchunks : 0;
  pl->g16 = pl->rows > 8;
  const int chunk0 =
      num_seqs < kMaxSeqsPerLaunch ? (num_seqs > 0 ? num_seqs : 1) : kMaxSeqsPerLaunch;
  // Two CTAs per SM (two independent pipelines) when their shared memory fits,
  // else one.  Keep at least 4 pipeline stages where possible by launching
  // fewer sequences at a time.
  bool ok = false;
  int chunk = chunk0;
  for (int occ = ctas_per_sm(D, pl->g16, BS, fp8); occ >= 1 && !ok; --occ) {
    int budget = di.smem_per_sm / occ - 1024;  // 1 KB per CTA is reserved by the system
    if (budget > di.max_smem) budget = di.max_smem;
    chunk = chunk0;
    for (;;) {
      // Bytes in flight per SM: past about 128 KB the memory system delivers no
      // more and a deeper ring measured slower (LLaMA-shaped batch, 8 KB pages, two
      // CTAs per SM: 8 stages 51.4 us, 10 52.2, 12 53.3); CTAs that cross many
      // (s, g) pieces gain from a deeper ring that absorbs the stall at each
      // piece end (ragged 256-sequence batch: 8 stages 617 us, 10 608).
      const long long pieces = (long long)chunk * H_kv * (pl->qchunks > 0 ? pl->qchunks : 1);
      const long long ring_cap =
          (pieces >= 2LL * di.sms * occ ? kRingBytesPerSmManyPieces : kRingBytesPerSm) / occ;
      if (plan_smem_any(D, BS, fp8, pl->rows, chunk, budget, ring_cap, pl->qchunks,
                        &pl->stages, &pl->smem) &&
          (pl->stages >= 4 || chunk <= 64)) {
        ok = true;
        pl->grid = di.sms * occ;
        break;
      }
      if (chunk <= 1) break;
      chunk = (chunk + 1) / 2;
    }
  }
  if (!ok) return PAGED_ATTN_ERR_SIZES;
  pl->chunk = chunk;
  // [0, 256): status word; then one combine counter per CTA of the largest grid
  // any launch on this device uses (two CTAs per SM); then the partial states.
  // The counter region depends on the device only (not on this launch's grid,
  // which is one CTA per SM for some shapes), so a workspace reused by calls of
  // any size always finds it zero: partials never land on it.
  pl->off_counters = kWsAlign;
  pl->off_partials = pl->off_counters + round_up((size_t)di.sms * 2 * 4, kWsAlign);
  pl->ws_bytes = pl->off_partials +
                 round_up((size_t)pl->grid * 2 * pl->rows * (size_t)(D + 4) * 4, kWsAlign);
  return PAGED_ATTN_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static cudaError_t cached_err = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cached_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                  cudaEnableDefault, &q);
    if (cached_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      cached = reinterpret_cast<EncodeTiledFn>(p);
    else if (cached_err == cudaSuccess)
      cached_err = cudaErrorSymbolNotFound;
  });
  if (!cached) return cuda_fail(cached_err);
  *fn = cached;
  return PAGED_ATTN_OK;
}

// 4-D view of a cache: (column within a 64-column half, row within a block =
// kv_head * BS + slot, half, block id).  A page of one KV head is the box
// {64, BS, D / 64, 1} at (0, g * BS, 0, block); it lands in shared memory as
// [half][row][128 bytes] with the 128-byte swizzle the kernel's ldmatrix
// addressing expects.
int encode_cache_map(const void* base, int D, int BS, int H_kv, long long num_blocks,
                     CUtensorMap* map, bool fp8 = false) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encoder(&enc);
  if (rc != PAGED_ATTN_OK) return rc;
  const int elem = fp8 ? 1 : 2;          // bytes per element
  const cuuint64_t inner = 128 / elem;   // elements in a 128-byte half of a row
  const cuuint64_t halves = (cuuint64_t)D * elem / 128;
  const cuuint64_t row_bytes = (cuuint64_t)D * elem;
  const cuuint64_t block_bytes = row_bytes * (cuuint64_t)H_kv * BS;
  cuuint64_t nb = (cuuint64_t)num_blocks;
  if (num_blocks <= 0) {
    // pool size unknown: any non-negative int32 block id is addressable, as long
    // as the described extent stays below 2^40 bytes
    nb = ((cuuint64_t)1 << 40) / block_bytes;
    if (nb > 0x7fffffffULL) nb = 0x7fffffffULL;
  }
  const cuuint64_t dims[4] = {inner, (cuuint64_t)H_kv * BS, halves, nb};
  const cuuint64_t strides[3] = {row_bytes, 128, block_bytes};
  const cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)BS, (cuuint32_t)halves, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail((int)r);
  return PAGED_ATTN_OK;
}

// x-packed caches.  A page of one KV head is contiguous in both (K [num_blocks,
// H_kv, D / 8, BS, 8], V [num_blocks, H_kv, D, BS]) and the kernel bulk-copies
// it, except V pages of 32 tokens, read through the 4-D view (BS, D, H_kv,
// block) of V: the box {BS, D, 1, 1} lands as [D][BS] with the 64-byte swizzle.
// The K map of the launch is unused and set to the same view.
int encode_xpacked_maps(const void* v, int D, int BS, int H_kv, long long num_blocks,
                        CUtensorMap* tk, CUtensorMap* tv) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encoder(&enc);
  if (rc != PAGED_ATTN_OK) return rc;
  const cuuint64_t head_bytes = (cuuint64_t)D * BS * 2;
  const cuuint64_t block_bytes = head_bytes * (cuuint64_t)H_kv;
  cuuint64_t nb = (cuuint64_t)num_blocks;
  if (num_blocks <= 0) {
    nb = ((cuuint64_t)1 << 40) / block_bytes;
    if (nb > 0x7fffffffULL) nb = 0x7fffffffULL;
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const cuuint64_t vdims[4] = {(cuuint64_t)BS, (cuuint64_t)D, (cuuint64_t)H_kv, nb};
  const cuuint64_t vstrides[3] = {(cuuint64_t)BS * 2, head_bytes, block_bytes};
  const cuuint32_t vbox[4] = {(cuuint32_t)BS, (cuuint32_t)D, 1, 1};
  CUresult r = enc(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v), vdims,
                   vstrides, vbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   BS == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail((int)r);
  *tk = *tv;
  return PAGED_ATTN_OK;
}

cudaError_t launch_dim(int D, int BS, bool g16, bool fp8, bool xp, const CUtensorMap& tk,
                       const CUtensorMap& tv, const DecodeParams& p, int grid, size_t smem,
                       cudaStream_t st) {
  if (p.qo_indptr != nullptr) {
    if (D == 64) return launch_decode_multi_d64(BS, g16, tk, tv, p, grid, smem, st);
    if (D == 128) return launch_decode_multi_d128(BS, g16, tk, tv, p, grid, smem, st);
    return launch_decode_multi_d256(BS, g16, tk, tv, p, grid, smem, st);
  }
  if (xp) {
    if (D == 64) return launch_decode_xp_d64(BS, g16, tk, tv, p, grid, smem, st);
    if (D == 128) return launch_decode_xp_d128(BS, g16, tk, tv, p, grid, smem, st);
    return launch_decode_xp_d256(BS, g16, tk, tv, p, grid, smem, st);
  }
  if (fp8)
    return D == 128 ? launch_decode_fp8_d128(BS, g16, tk, tv, p, grid, smem, st)
                    : launch_decode_fp8_d256(BS, g16, tk, tv, p, grid, smem, st);
  if (D == 64) return launch_decode_d64(BS, g16, tk, tv, p, grid, smem, st);
  if (D == 128) return launch_decode_d128(BS, g16, tk, tv, p, grid, smem, st);
  return launch_decode_d256(BS, g16, tk, tv, p, grid, smem, st);
}

int check_pointers(const void* q, const void* k, const void* v, const void* out,
                   const int32_t* bt, const int32_t* sl) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(bt) ||
      !aligned16(sl))
    return PAGED_ATTN_ERR_POINTER;
  return PAGED_ATTN_OK;
}

// Runs the whole operation in chunks of plan.chunk sequences on `stream`.
// With k_new / v_new (else null), each sequence's new token is first written
// into the caches by the decode kernel itself (fused cache append).
int run(const Plan& pl, const void* q, const void* k_cache, const void* v_cache, void* out,
        const int32_t* bt, const int32_t* seq_lens, int num_seqs, int H_q, int H_kv,
        int max_blocks_per_seq, float scale, void* ws, int32_t* status, long long num_blocks,
        cudaStream_t stream, const void* k_new = nullptr, const void* v_new = nullptr,
        const float* k_scale = nullptr, const float* v_scale = nullptr,
        const int32_t* qo_indptr = nullptr, int total_q = 0) {
  CUtensorMap tk, tv;
  int rc;
  if (pl.xp) {
    rc = encode_xpacked_maps(v_cache, pl.D, pl.BS, H_kv, num_blocks, &tk, &tv);
    if (rc != PAGED_ATTN_OK) return rc;
  } else {
    rc = encode_cache_map(k_cache, pl.D, pl.BS, H_kv, num_blocks, &tk, pl.fp8);
    if (rc != PAGED_ATTN_OK) return rc;
    rc = encode_cache_map(v_cache, pl.D, pl.BS, H_kv, num_blocks, &tv, pl.fp8);
    if (rc != PAGED_ATTN_OK) return rc;
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  for (int s0 = 0; s0 < num_seqs; s0 += pl.chunk) {
    const int n = num_seqs - s0 < pl.chunk ? num_seqs - s0 : pl.chunk;
    DecodeParams p;
    // multi-token decode: q and out rows are found through qo_indptr (absolute)
    const size_t row0 = qo_indptr ? 0 : (size_t)s0;
    p.q = static_cast<const __nv_bfloat16*>(q) + row0 * H_q * pl.D;
    p.out = static_cast<__nv_bfloat16*>(out) + row0 * H_q * pl.D;
    p.qo_indptr = qo_indptr ? qo_indptr + s0 : nullptr;
    p.rows = pl.rows;
    p.chunks = pl.qchunks > 0 ? pl.qchunks : 1;
    p.total_q = total_q;
    p.block_tables = bt + (size_t)s0 * max_blocks_per_seq;
    p.seq_lens = seq_lens + s0;
    p.num_seqs = n;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = pl.G;
    p.maxb = max_blocks_per_seq;
    p.stages = pl.stages;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = status ? status : reinterpret_cast<int32_t*>(wsb);
    p.counters = reinterpret_cast<int32_t*>(wsb + pl.off_counters);
    p.partials = reinterpret_cast<float*>(wsb + pl.off_partials);
    p.num_blocks = num_blocks;
    p.early = (g_launch_flags & PAGED_ATTN_FLAG_EARLY_PROLOGUE) ? 1 : 0;
    p.k_new = k_new ? static_cast<const __nv_bfloat16*>(k_new) + (size_t)s0 * H_kv * pl.D
                    : nullptr;
    p.v_new = v_new ? static_cast<const __nv_bfloat16*>(v_new) + (size_t)s0 * H_kv * pl.D
                    : nullptr;
    p.k_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(k_cache));
    p.v_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(v_cache));
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    cudaError_t e =
        launch_dim(pl.D, pl.BS, pl.g16, pl.fp8, pl.xp, tk, tv, p, pl.grid, pl.smem, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PAGED_ATTN_OK;
}

// The library-owned workspace of the current device, grown to at least `bytes`.
int owned_workspace(size_t bytes, cudaStream_t stream, void** out) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != PAGED_ATTN_OK) return rc;
  cudaError_t e;
  std::lock_guard<std::mutex> lk(g_mu);
  OwnedWorkspace& w = g_ws[dev];
  if (w.bytes < bytes) {
    if (w.ptr) {
      // earlier calls on any stream may still use the old buffer
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    void* p = nullptr;
    if ((e = cudaMalloc(&p, bytes)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemsetAsync(p, 0, bytes, stream)) != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(e);
    }
    w.ptr = p;
    w.bytes = bytes;
  }
  *out = w.ptr;
  return PAGED_ATTN_OK;
}

// Scratch for paged_attn_decode_static: a fixed array every GPU that loads the
// library holds until the process exits, so that entry point never allocates.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device, looked up once per
// device (in host code the array's name is only a stand-in, not an address).
int static_scratch_address(void** out) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != PAGED_ATTN_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_static_scratch_ptr[dev] != nullptr) {
    *out = g_static_scratch_ptr[dev];
    return PAGED_ATTN_OK;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e);
  g_static_scratch_ptr[dev] = ptr;
  *out = ptr;
  return PAGED_ATTN_OK;
}

int common_checks(const void* q, const void* k, const void* v, const void* out, const int32_t* bt,
                  const int32_t* sl, int num_seqs, int H_q, int H_kv, int head_dim,
                  int max_blocks_per_seq, int block_size, float scale) {
  int rc = validate_sizes(num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK) return rc;
  if (!std::isfinite(scale)) return PAGED_ATTN_ERR_SCALE;
  if (num_seqs == 0) return PAGED_ATTN_OK;
  return check_pointers(q, k, v, out, bt, sl);
}

}  // namespace
}  // namespace pagedattn

using namespace pagedattn;

extern "C" {

int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int H_q, int H_kv, int head_dim, int max_blocks_per_seq, int block_size,
                      float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st);
}

int paged_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache, void* out,
                            const int32_t* qo_indptr, const int32_t* block_tables,
                            const int32_t* seq_lens, int num_seqs, int total_q, int max_q_len,
                            int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                            int block_size, float scale, void* stream) {
  int rc = validate_sizes(num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK) return rc;
  if (!std::isfinite(scale)) return PAGED_ATTN_ERR_SCALE;
  const int G = H_q / H_kv;
  if (total_q < 0 || max_q_len < 1 || (long long)max_q_len * G > kMaxMultiRows ||
      (long long)total_q * H_q * head_dim >= (1LL << 40))
    return PAGED_ATTN_ERR_SIZES;
  if (num_seqs == 0) return PAGED_ATTN_OK;
  rc = check_pointers(q, k_cache, v_cache, out, block_tables, seq_lens);
  if (rc != PAGED_ATTN_OK) return rc;
  if (!aligned16(qo_indptr)) return PAGED_ATTN_ERR_POINTER;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  // one n8 MMA tile of rows when a KV head's q_len * G rows fit, else pieces of 16
  const int rows = max_q_len * G <= 8 ? 8 : 16;
  const int qchunks = (max_q_len * G + rows - 1) / rows;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl, false, rows,
                      qchunks)) != PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st, nullptr, nullptr, nullptr, nullptr,
             qo_indptr, total_q);
}

int paged_attn_decode_xpacked(const void* q, const void* k_cache, const void* v_cache, void* out,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                              int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                              int block_size, float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  pl.xp = true;  // same shared-memory plan as the bf16 layout
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st);
}

int paged_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale, void* out,
                          const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                          int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                          int block_size, float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK) return rc;
  if (head_dim == 64) return PAGED_ATTN_ERR_HEAD_DIM;  // FP8 pages need 128-byte rows
  if (num_seqs == 0) return PAGED_ATTN_OK;
  if (!aligned16(k_scale) || !aligned16(v_scale)) return PAGED_ATTN_ERR_POINTER;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl, true)) !=
      PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st, nullptr, nullptr, k_scale, v_scale);
}

int paged_attn_append_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, void* out, const int32_t* block_tables,
                             const int32_t* seq_lens, int num_seqs, int H_q, int H_kv,
                             int head_dim, int max_blocks_per_seq, int block_size, float scale,
                             void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (!aligned16(k_new) || !aligned16(v_new)) return PAGED_ATTN_ERR_POINTER;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  // Fused, the warp that reads a piece's last page patches the new rows into it,
  // a small cost per piece on that CTA's path.  When CTAs average kAppendApartPieces
  // or more (s, g) pieces, the CTA crossing the most short sequences sets the
  // kernel's end and a separate append launch ahead of the decode is cheaper
  // (ragged 256-sequence batch: decode 619 us, fused 630, apart 622; LLaMA-shaped
  // batch: decode 51.3, fused 51.6, apart 53.4).  Both give the same bits.
  if ((long long)num_seqs * H_kv >= (long long)kAppendApartPieces * pl.grid) {
    AppendParams a;
    a.k_new = static_cast<const __nv_bfloat16*>(k_new);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new);
    a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.H_kv = H_kv;
    a.D = head_dim;
    a.maxb = max_blocks_per_seq;
    a.BS = block_size;
    a.num_blocks = 0;
    cudaError_t e = launch_append(a, di.sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
               max_blocks_per_seq, scale, ws, nullptr, 0, st);
  }
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st, k_new, v_new);
}

int paged_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int H_kv,
                    int head_dim, int max_blocks_per_seq, int block_size, void* stream) {
  // the decode's size rules with a one-head query group
  int rc = validate_sizes(num_seqs, H_kv, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(block_tables) || !aligned16(seq_lens))
    return PAGED_ATTN_ERR_POINTER;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  AppendParams a;
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.H_kv = H_kv;
  a.D = head_dim;
  a.maxb = max_blocks_per_seq;
  a.BS = block_size;
  a.num_blocks = 0;
  cudaError_t e = launch_append(a, di.sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PAGED_ATTN_OK : cuda_fail(e);
}

size_t paged_attn_workspace_bytes(int num_seqs, int H_q, int H_kv, int head_dim,
                                  int max_blocks_per_seq, int block_size) {
  if (validate_sizes(num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size) !=
      PAGED_ATTN_OK)
    return 0;
  DeviceInfo di;
  if (device_info(&di) != PAGED_ATTN_OK) return 0;
  Plan pl;
  if (make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl) != PAGED_ATTN_OK) return 0;
  return pl.ws_bytes;
}

int paged_attn_decode_ws(const void* q, const void* k_cache, const void* v_cache, void* out,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                         int H_q, int H_kv, int head_dim, int max_blocks_per_seq, int block_size,
                         float scale, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) != 0)
    return PAGED_ATTN_ERR_WORKSPACE;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  if (workspace_bytes < pl.ws_bytes) return PAGED_ATTN_ERR_WORKSPACE;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, workspace, nullptr, 0, static_cast<cudaStream_t>(stream));
}

int paged_attn_decode_checked(const void* q, const void* k_cache, const void* v_cache, void* out,
                              const int32_t* block_tables, const int32_t* seq_lens,
                              int num_seqs, int H_q, int H_kv, int head_dim,
                              int max_blocks_per_seq, int block_size, float scale,
                              long long num_blocks, int32_t* d_status, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (num_blocks <= 0 || num_blocks > 0x7fffffffLL) return PAGED_ATTN_ERR_SIZES;
  if (d_status == nullptr || (reinterpret_cast<uintptr_t>(d_status) & 3) != 0)
    return PAGED_ATTN_ERR_POINTER;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((rc = owned_workspace(pl.ws_bytes, st, &ws)) != PAGED_ATTN_OK) return rc;
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, d_status, num_blocks, st);
}

int paged_attn_decode_static(const void* q, const void* k_cache, const void* v_cache, void* out,
                             const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                             int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                             int block_size, float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  DeviceInfo di;
  if ((rc = device_info(&di)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(num_seqs, H_q, H_kv, head_dim, block_size, di, &pl)) != PAGED_ATTN_OK)
    return rc;
  if (pl.ws_bytes > kStaticScratchBytes) return PAGED_ATTN_ERR_STATIC_SCRATCH;
  void* ws = nullptr;
  if ((rc = static_scratch_address(&ws)) != PAGED_ATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left; the status word and the
  // combine counters must start at zero.
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.off_partials, st);
  if (e != cudaSuccess) return cuda_fail(e);
  return run(pl, q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
             max_blocks_per_seq, scale, ws, nullptr, 0, st);
}

const char* paged_attn_status_string(int status) {
  switch (status) {
    case PAGED_ATTN_OK: return "ok";
    case PAGED_ATTN_ERR_POINTER: return "null or misaligned pointer";
    case PAGED_ATTN_ERR_HEADS: return "H_q must be a positive multiple of H_kv with H_q/H_kv <= 16";
    case PAGED_ATTN_ERR_HEAD_DIM: return "head_dim must be 64, 128 or 256";
    case PAGED_ATTN_ERR_BLOCK_SIZE: return "block_size must be 16 or 32";
    case PAGED_ATTN_ERR_SIZES: return "num_seqs, max_blocks_per_seq or num_blocks out of range";
    case PAGED_ATTN_ERR_CUDA: return "CUDA call failed (see paged_attn_last_cuda_error)";
    case PAGED_ATTN_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case PAGED_ATTN_ERR_SCALE: return "scale is not finite";
    case PAGED_ATTN_ERR_STATIC_SCRATCH:
      return "sizes need more scratch than paged_attn_decode_static's fixed 4 MiB array";
    case PAGED_ATTN_ERR_FLAGS: return "unknown launch flag bits";
    default: return "unknown status";
  }
}

int paged_attn_set_launch_flags(int flags) {
  if (flags & ~PAGED_ATTN_FLAG_EARLY_PROLOGUE) return PAGED_ATTN_ERR_FLAGS;
  g_launch_flags = flags;
  return PAGED_ATTN_OK;
}

int paged_attn_last_cuda_error(void) { return g_last_cuda_error; }

int paged_attn_version(void) { return 100; }

}  // extern "C"
