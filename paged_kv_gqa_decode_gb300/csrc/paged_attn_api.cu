// C ABI of the paged-KV GQA decode library (include/paged_attn.h): argument
// validation, launch planning (grid, pipeline depth, workspace), TMA tensor
// maps, and the per-device workspace the plain entry point owns.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
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
// paged_attn_set_checks: pool size and device status word for every call of
// this thread (0 / null: no checks)
thread_local long long g_check_blocks = 0;
thread_local int32_t* g_check_status = nullptr;
#ifdef PAGED_ATTN_WAIT_TEST
thread_local int g_test_skip_unit = -1;
thread_local int g_test_skip_publish = 0;
#endif

constexpr int kMaxSeqsPerLaunch = 4096;
constexpr size_t kWsAlign = 256;
constexpr int kAppendApartPieces = 4;  // (s, g) pieces per CTA from which the append runs apart
constexpr int kMaxMultiRows = 256;      // multi-token decode: max q_len * G (16 pieces of 16 rows)
constexpr long long kRingBytesPerSm = 128 << 10;            // K/V rings of one SM, few pieces per CTA
constexpr long long kRingBytesPerSmManyPieces = 160 << 10;  // ... two or more pieces per CTA
constexpr long long kRingBytesPerSmThreeCtas = 150 << 10;   // three FP8 CTAs: 12 stages each

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

int device_info(DeviceInfo* out, int* dev_out = nullptr) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != PAGED_ATTN_OK) return rc;
  if (dev_out) *dev_out = dev;
  thread_local DeviceInfo tl_info[kMaxDevices];  // this thread's copy of g_info
  if (tl_info[dev].sms > 0) {
    *out = tl_info[dev];
    return PAGED_ATTN_OK;
  }
  cudaError_t e;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_info[dev].sms > 0) {
    *out = tl_info[dev] = g_info[dev];
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
  g_info[dev] = tl_info[dev] = di;
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
      // Three FP8 CTAs per SM: 12 stages each (8 measured slower on the
      // LLaMA-shaped batch, 32.7 against 31.0 us; 16 do not fit).
      const long long pieces = (long long)chunk * H_kv * (pl->qchunks > 0 ? pl->qchunks : 1);
      const long long ring_cap =
          (occ >= 3                           ? kRingBytesPerSmThreeCtas
           : pieces >= 2LL * di.sms * occ ? kRingBytesPerSmManyPieces
                                          : kRingBytesPerSm) /
          occ;
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
  // any launch on this device uses (kMaxCtasPerSm CTAs per SM); then the
  // partial states.
  // The counter region depends on the device only (not on this launch's grid,
  // which is one CTA per SM for some shapes), so a workspace reused by calls of
  // any size always finds it zero: partials never land on it.
  pl->off_counters = kWsAlign;
  pl->off_partials = pl->off_counters + round_up((size_t)di.sms * kMaxCtasPerSm * 4, kWsAlign);
  pl->ws_bytes = pl->off_partials +
                 round_up((size_t)pl->grid * 2 * pl->rows * (size_t)(D + 4) * 4, kWsAlign);
  return PAGED_ATTN_OK;
}

// make_plan through a small per-thread cache: the plan depends only on the
// sizes, the variant and the device, so a decode loop plans once.
int cached_plan(int num_seqs, int H_q, int H_kv, int D, int BS, int dev, const DeviceInfo& di,
                Plan* pl, bool fp8 = false, int rows = 0, int qchunks = 0) {
  struct Entry {
    int key[9];
    Plan plan;
    bool used;
  };
  constexpr int kEntries = 16;
  thread_local Entry tl_plans[kEntries] = {};
  const int key[9] = {num_seqs, H_q, H_kv, D, BS, fp8 ? 1 : 0, rows, qchunks, dev};
  uint32_t h = 2166136261u;
  for (int k : key) h = (h ^ (uint32_t)k) * 16777619u;
  Entry& e = tl_plans[h % kEntries];
  if (e.used && std::memcmp(e.key, key, sizeof key) == 0) {
    *pl = e.plan;
    return PAGED_ATTN_OK;
  }
  int rc = make_plan(num_seqs, H_q, H_kv, D, BS, di, pl, fp8, rows, qchunks);
  if (rc != PAGED_ATTN_OK) return rc;
  std::memcpy(e.key, key, sizeof key);
  e.plan = *pl;
  e.used = true;
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
#ifdef PAGED_ATTN_WAIT_TEST
  // the test build carries the single-token bf16 head_dim-128 kernels only
  if (p.qo_indptr != nullptr || xp || fp8 || D != 128) return cudaErrorNotSupported;
  return launch_decode_d128(BS, g16, tk, tv, p, grid, smem, st);
#endif
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

// The tensor maps of a call through a per-thread direct-mapped cache: a map
// depends only on the base address and the sizes it describes, so a decode
// loop over the same caches encodes each once.
enum MapKind { kMapBf16 = 0, kMapFp8 = 1, kMapXpackedV = 2 };

int cached_map(const void* base, int D, int BS, int H_kv, long long num_blocks, MapKind kind,
               CUtensorMap* out) {
  struct Entry {
    CUtensorMap map;
    const void* base;
    long long num_blocks;
    int D, BS, H_kv, kind;
    bool used;
  };
  constexpr int kEntries = 256;
  thread_local std::unique_ptr<Entry[]> tl_maps;
  if (!tl_maps) tl_maps.reset(new Entry[kEntries]());
  const uint64_t a = reinterpret_cast<uintptr_t>(base);
  const uint64_t h = (a >> 8) * 0x9E3779B97F4A7C15ull ^ ((uint64_t)kind << 1) ^
                     ((uint64_t)D * 31 + (uint64_t)BS * 7 + (uint64_t)H_kv);
  Entry& e = tl_maps[(h >> 32) % kEntries];
  if (e.used && e.base == base && e.num_blocks == num_blocks && e.D == D && e.BS == BS &&
      e.H_kv == H_kv && e.kind == kind) {
    *out = e.map;
    return PAGED_ATTN_OK;
  }
  CUtensorMap m;
  int rc;
  if (kind == kMapXpackedV) {
    CUtensorMap unused;
    rc = encode_xpacked_maps(base, D, BS, H_kv, num_blocks, &unused, &m);
  } else {
    rc = encode_cache_map(base, D, BS, H_kv, num_blocks, &m, kind == kMapFp8);
  }
  if (rc != PAGED_ATTN_OK) return rc;
  e.map = m;
  e.base = base;
  e.num_blocks = num_blocks;
  e.D = D;
  e.BS = BS;
  e.H_kv = H_kv;
  e.kind = kind;
  e.used = true;
  *out = m;
  return PAGED_ATTN_OK;
}

// Everything one decode call hands to its launches.
struct Operands {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  void* out;
  const int32_t* bt;
  const int32_t* seq_lens;
  int num_seqs, H_q, H_kv, maxb;
  float scale;
  void* ws;                         // workspace (status word, counters, partials)
  int32_t* status = nullptr;        // caller status word (null: the workspace's)
  long long num_blocks = 0;         // > 0: block ids checked against the pool
  bool early = false;               // early-prologue launch (caller's guarantee holds)
  const void* k_new = nullptr;      // fused cache append (bf16)
  const void* v_new = nullptr;
  const float* k_scale = nullptr;   // FP8 row floats
  const float* v_scale = nullptr;
  const int32_t* qo_indptr = nullptr;  // multi-token decode
  int total_q = 0;
  int causal = 1;
};

// The calling thread's device-side checks (paged_attn_set_checks), if any.
void apply_checks(Operands* o) {
  if (g_check_blocks > 0) {
    o->num_blocks = g_check_blocks;
    o->status = g_check_status;
  }
}

// The early prologue applies when the caller asked for it on this thread and
// nothing the library itself launched just before writes what the producer
// reads ahead of the wait.
bool early_requested() { return (g_launch_flags & PAGED_ATTN_FLAG_EARLY_PROLOGUE) != 0; }

// Runs the whole operation in chunks of plan.chunk sequences on `stream`.
int run(const Plan& pl, const Operands& o, cudaStream_t stream) {
  CUtensorMap tk, tv;
  int rc;
  if (pl.xp) {
    rc = cached_map(o.v_cache, pl.D, pl.BS, o.H_kv, o.num_blocks, kMapXpackedV, &tv);
    if (rc != PAGED_ATTN_OK) return rc;
    tk = tv;  // unused by the x-packed kernel
  } else {
    const MapKind kind = pl.fp8 ? kMapFp8 : kMapBf16;
    rc = cached_map(o.k_cache, pl.D, pl.BS, o.H_kv, o.num_blocks, kind, &tk);
    if (rc != PAGED_ATTN_OK) return rc;
    rc = cached_map(o.v_cache, pl.D, pl.BS, o.H_kv, o.num_blocks, kind, &tv);
    if (rc != PAGED_ATTN_OK) return rc;
  }
  uint8_t* wsb = static_cast<uint8_t*>(o.ws);
  for (int s0 = 0; s0 < o.num_seqs; s0 += pl.chunk) {
    const int n = o.num_seqs - s0 < pl.chunk ? o.num_seqs - s0 : pl.chunk;
    DecodeParams p;
    // multi-token decode: q and out rows are found through qo_indptr (absolute)
    const size_t row0 = o.qo_indptr ? 0 : (size_t)s0;
    p.q = static_cast<const __nv_bfloat16*>(o.q) + row0 * o.H_q * pl.D;
    p.out = static_cast<__nv_bfloat16*>(o.out) + row0 * o.H_q * pl.D;
    p.qo_indptr = o.qo_indptr ? o.qo_indptr + s0 : nullptr;
    p.rows = pl.rows;
    p.chunks = pl.qchunks > 0 ? pl.qchunks : 1;
    p.total_q = o.total_q;
    p.causal = o.causal;
    p.block_tables = o.bt + (size_t)s0 * o.maxb;
    p.seq_lens = o.seq_lens + s0;
    p.num_seqs = n;
    p.H_q = o.H_q;
    p.H_kv = o.H_kv;
    p.G = pl.G;
    p.maxb = o.maxb;
    p.stages = pl.stages;
    p.scale_log2 = o.scale * 1.4426950408889634f;
    p.status = o.status ? o.status : reinterpret_cast<int32_t*>(wsb);
    p.counters = reinterpret_cast<int32_t*>(wsb + pl.off_counters);
    p.partials = reinterpret_cast<float*>(wsb + pl.off_partials);
    p.num_blocks = o.num_blocks;
    p.early = o.early ? 1 : 0;
    p.k_new = o.k_new ? static_cast<const __nv_bfloat16*>(o.k_new) + (size_t)s0 * o.H_kv * pl.D
                      : nullptr;
    p.v_new = o.v_new ? static_cast<const __nv_bfloat16*>(o.v_new) + (size_t)s0 * o.H_kv * pl.D
                      : nullptr;
    p.k_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(o.k_cache));
    p.v_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(o.v_cache));
    p.k_scale = o.k_scale;
    p.v_scale = o.v_scale;
#ifdef PAGED_ATTN_WAIT_TEST
    p.test_skip_unit = g_test_skip_unit;
    p.test_skip_publish = g_test_skip_publish;
#endif
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
      // Earlier calls on this stream may still use the old buffer: free it in
      // stream order (calls on other streams overlapping this one race on the
      // shared workspace anyway, as the header says).  No device-wide sync.
      if ((e = cudaFreeAsync(w.ptr, stream)) != cudaSuccess) return cuda_fail(e);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    void* p = nullptr;
    // stream-ordered, like the release of the old one (the device's default pool)
    if ((e = cudaMallocAsync(&p, bytes, stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemsetAsync(p, 0, bytes, stream)) != cudaSuccess) {
      cudaFreeAsync(p, stream);
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

// A decode call's operands with the caller's pointers and sizes.
Operands operands(const void* q, const void* k_cache, const void* v_cache, void* out,
                  const int32_t* bt, const int32_t* sl, int num_seqs, int H_q, int H_kv,
                  int max_blocks_per_seq, float scale) {
  Operands o;
  o.q = q;
  o.k_cache = k_cache;
  o.v_cache = v_cache;
  o.out = out;
  o.bt = bt;
  o.seq_lens = sl;
  o.num_seqs = num_seqs;
  o.H_q = H_q;
  o.H_kv = H_kv;
  o.maxb = max_blocks_per_seq;
  o.scale = scale;
  o.ws = nullptr;
  return o;
}

// Plans a decode launch on the current device and runs it in the library-owned
// workspace (o.ws null) or the one given.  rows > 0: multi-token pieces.
int plan_and_run(Operands& o, int head_dim, int block_size, bool fp8, bool xp, int rows,
                 int qchunks, cudaStream_t st) {
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(&di, &dev);
  if (rc != PAGED_ATTN_OK) return rc;
  Plan pl;
  rc = cached_plan(o.num_seqs, o.H_q, o.H_kv, head_dim, block_size, dev, di, &pl, fp8, rows,
                   qchunks);
  if (rc != PAGED_ATTN_OK) return rc;
  pl.xp = xp;  // same shared-memory plan as the bf16 layout
  if (o.ws == nullptr && (rc = owned_workspace(pl.ws_bytes, st, &o.ws)) != PAGED_ATTN_OK)
    return rc;
  return run(pl, o, st);
}

AppendParams append_params(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const int32_t* bt, const int32_t* sl, int num_seqs, int H_kv,
                           int head_dim, int max_blocks_per_seq, int block_size) {
  AppendParams a;
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = nullptr;
  a.v_scale = nullptr;
  a.block_tables = bt;
  a.seq_lens = sl;
  a.qo_indptr = nullptr;
  a.num_seqs = num_seqs;
  a.total_q = 0;
  a.H_kv = H_kv;
  a.D = head_dim;
  a.maxb = max_blocks_per_seq;
  a.BS = block_size;
  a.num_blocks = g_check_blocks;
  a.status = g_check_blocks > 0 ? g_check_status : nullptr;
  return a;
}

int sms_of_device(int* sms) {
  DeviceInfo di;
  int rc = device_info(&di);
  if (rc == PAGED_ATTN_OK) *sms = di.sms;
  return rc;
}

int multi_checks(const void* q, const void* k_cache, const void* v_cache, const void* out,
                 const int32_t* qo_indptr, const int32_t* bt, const int32_t* sl, int num_seqs,
                 int total_q, int max_q_len, int H_q, int H_kv, int head_dim,
                 int max_blocks_per_seq, int block_size, float scale) {
  int rc = validate_sizes(num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK) return rc;
  if (!std::isfinite(scale)) return PAGED_ATTN_ERR_SCALE;
  const int G = H_q / H_kv;
  if (total_q < 0 || max_q_len < 1 || (long long)max_q_len * G > kMaxMultiRows ||
      (long long)total_q * H_q * head_dim >= (1LL << 40))
    return PAGED_ATTN_ERR_SIZES;
  if (num_seqs == 0) return PAGED_ATTN_OK;
  rc = check_pointers(q, k_cache, v_cache, out, bt, sl);
  if (rc != PAGED_ATTN_OK) return rc;
  if (!aligned16(qo_indptr)) return PAGED_ATTN_ERR_POINTER;
  return PAGED_ATTN_OK;
}

int decode_multi_impl(const void* q, const void* k_cache, const void* v_cache, void* out,
                      const int32_t* qo_indptr, const int32_t* bt, const int32_t* sl,
                      int num_seqs, int total_q, int max_q_len, int H_q, int H_kv, int head_dim,
                      int max_blocks_per_seq, int block_size, float scale, int causal, bool early,
                      cudaStream_t st) {
  Operands o = operands(q, k_cache, v_cache, out, bt, sl, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.qo_indptr = qo_indptr;
  o.total_q = total_q;
  o.causal = causal ? 1 : 0;
  o.early = early;
  apply_checks(&o);
  // one n8 MMA tile of rows when a KV head's q_len * G rows fit, else pieces of 16
  const int G = H_q / H_kv;
  const int rows = max_q_len * G <= 8 ? 8 : 16;
  const int qchunks = (max_q_len * G + rows - 1) / rows;
  return plan_and_run(o, head_dim, block_size, false, false, rows, qchunks, st);
}

int fp8_checks(const void* q, const void* k8, const void* v8, const void* k_scale,
               const void* v_scale, const void* out, const int32_t* bt, const int32_t* sl,
               int num_seqs, int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
               int block_size, float scale) {
  int rc = common_checks(q, k8, v8, out, bt, sl, num_seqs, H_q, H_kv, head_dim,
                         max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK) return rc;
  if (head_dim == 64) return PAGED_ATTN_ERR_HEAD_DIM;  // FP8 pages need 128-byte rows
  if (num_seqs == 0) return PAGED_ATTN_OK;
  if (!aligned16(k_scale) || !aligned16(v_scale)) return PAGED_ATTN_ERR_POINTER;
  return PAGED_ATTN_OK;
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
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.early = early_requested();
  apply_checks(&o);
  return plan_and_run(o, head_dim, block_size, false, false, 0, 0,
                      static_cast<cudaStream_t>(stream));
}

int paged_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache, void* out,
                            const int32_t* qo_indptr, const int32_t* block_tables,
                            const int32_t* seq_lens, int num_seqs, int total_q, int max_q_len,
                            int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                            int block_size, float scale, void* stream) {
  return paged_attn_decode_multi_ex(q, k_cache, v_cache, out, qo_indptr, block_tables, seq_lens,
                                    num_seqs, total_q, max_q_len, H_q, H_kv, head_dim,
                                    max_blocks_per_seq, block_size, scale, 1, stream);
}

int paged_attn_decode_multi_ex(const void* q, const void* k_cache, const void* v_cache,
                               void* out, const int32_t* qo_indptr, const int32_t* block_tables,
                               const int32_t* seq_lens, int num_seqs, int total_q, int max_q_len,
                               int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                               int block_size, float scale, int is_causal, void* stream) {
  int rc = multi_checks(q, k_cache, v_cache, out, qo_indptr, block_tables, seq_lens, num_seqs,
                        total_q, max_q_len, H_q, H_kv, head_dim, max_blocks_per_seq, block_size,
                        scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  return decode_multi_impl(q, k_cache, v_cache, out, qo_indptr, block_tables, seq_lens, num_seqs,
                           total_q, max_q_len, H_q, H_kv, head_dim, max_blocks_per_seq,
                           block_size, scale, is_causal, early_requested(),
                           static_cast<cudaStream_t>(stream));
}

int paged_attn_decode_xpacked(const void* q, const void* k_cache, const void* v_cache, void* out,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                              int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                              int block_size, float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.early = early_requested();
  apply_checks(&o);
  return plan_and_run(o, head_dim, block_size, false, true, 0, 0,
                      static_cast<cudaStream_t>(stream));
}

int paged_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale, void* out,
                          const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                          int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                          int block_size, float scale, void* stream) {
  int rc = fp8_checks(q, k_cache, v_cache, k_scale, v_scale, out, block_tables, seq_lens,
                      num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.k_scale = k_scale;
  o.v_scale = v_scale;
  o.early = early_requested();
  apply_checks(&o);
  return plan_and_run(o, head_dim, block_size, true, false, 0, 0,
                      static_cast<cudaStream_t>(stream));
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
  int dev = 0;
  DeviceInfo di;
  if ((rc = device_info(&di, &dev)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = cached_plan(num_seqs, H_q, H_kv, head_dim, block_size, dev, di, &pl)) !=
      PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  apply_checks(&o);
  if ((rc = owned_workspace(pl.ws_bytes, st, &o.ws)) != PAGED_ATTN_OK) return rc;
  // Fused, the warp that reads a piece's last page patches the new rows into it,
  // a small cost per piece on that CTA's path.  When CTAs average kAppendApartPieces
  // or more (s, g) pieces, the CTA crossing the most short sequences sets the
  // kernel's end and a separate append launch ahead of the decode is cheaper
  // (ragged 256-sequence batch: decode 619 us, fused 630, apart 622; LLaMA-shaped
  // batch: decode 51.3, fused 51.6, apart 53.4).  Both give the same bits.
  if ((long long)num_seqs * H_kv >= (long long)kAppendApartPieces * pl.grid) {
    AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                   num_seqs, H_kv, head_dim, max_blocks_per_seq, block_size);
    cudaError_t e = launch_append(a, di.sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    // The append just written is what the decode's producer reads first: the
    // decode waits for it before any global access (no early prologue).
    o.early = false;
    return run(pl, o, st);
  }
  // Fused: the new rows are patched into the pages in shared memory, whatever
  // the producer's copy brought, so the early prologue stays as requested.
  o.early = early_requested();
  o.k_new = k_new;
  o.v_new = v_new;
  return run(pl, o, st);
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
  int sms = 0;
  if ((rc = sms_of_device(&sms)) != PAGED_ATTN_OK) return rc;
  AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                 H_kv, head_dim, max_blocks_per_seq, block_size);
  cudaError_t e = launch_append(a, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PAGED_ATTN_OK : cuda_fail(e);
}

int paged_kv_append_multi(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int32_t* qo_indptr, const int32_t* block_tables,
                          const int32_t* seq_lens, int num_seqs, int total_q, int H_kv,
                          int head_dim, int max_blocks_per_seq, int block_size, void* stream) {
  int rc = validate_sizes(num_seqs, H_kv, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK) return rc;
  if (total_q < 0 || (long long)total_q * H_kv * head_dim >= (1LL << 40))
    return PAGED_ATTN_ERR_SIZES;
  if (num_seqs == 0 || total_q == 0) return PAGED_ATTN_OK;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(qo_indptr) || !aligned16(block_tables) || !aligned16(seq_lens))
    return PAGED_ATTN_ERR_POINTER;
  int sms = 0;
  if ((rc = sms_of_device(&sms)) != PAGED_ATTN_OK) return rc;
  AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                 H_kv, head_dim, max_blocks_per_seq, block_size);
  a.qo_indptr = qo_indptr;
  a.total_q = total_q;
  cudaError_t e = launch_append(a, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PAGED_ATTN_OK : cuda_fail(e);
}

int paged_attn_append_decode_multi(const void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, void* out,
                                   const int32_t* qo_indptr, const int32_t* block_tables,
                                   const int32_t* seq_lens, int num_seqs, int total_q,
                                   int max_q_len, int H_q, int H_kv, int head_dim,
                                   int max_blocks_per_seq, int block_size, float scale,
                                   int is_causal, void* stream) {
  int rc = multi_checks(q, k_cache, v_cache, out, qo_indptr, block_tables, seq_lens, num_seqs,
                        total_q, max_q_len, H_q, H_kv, head_dim, max_blocks_per_seq, block_size,
                        scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (!aligned16(k_new) || !aligned16(v_new)) return PAGED_ATTN_ERR_POINTER;
  int sms = 0;
  if ((rc = sms_of_device(&sms)) != PAGED_ATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (total_q > 0) {
    AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                   num_seqs, H_kv, head_dim, max_blocks_per_seq, block_size);
    a.qo_indptr = qo_indptr;
    a.total_q = total_q;
    cudaError_t e = launch_append(a, sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // the decode reads the rows just appended: plain launch (no early prologue)
  return decode_multi_impl(q, k_cache, v_cache, out, qo_indptr, block_tables, seq_lens, num_seqs,
                           total_q, max_q_len, H_q, H_kv, head_dim, max_blocks_per_seq,
                           block_size, scale, is_causal, false, st);
}

int paged_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        float* k_scale, float* v_scale, const int32_t* block_tables,
                        const int32_t* seq_lens, int num_seqs, int H_kv, int head_dim,
                        int max_blocks_per_seq, int block_size, void* stream) {
  int rc = validate_sizes(num_seqs, H_kv, H_kv, head_dim, max_blocks_per_seq, block_size);
  if (rc != PAGED_ATTN_OK) return rc;
  if (head_dim == 64) return PAGED_ATTN_ERR_HEAD_DIM;  // as the FP8 decode
  if (num_seqs == 0) return PAGED_ATTN_OK;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_scale) || !aligned16(v_scale) || !aligned16(block_tables) ||
      !aligned16(seq_lens))
    return PAGED_ATTN_ERR_POINTER;
  int sms = 0;
  if ((rc = sms_of_device(&sms)) != PAGED_ATTN_OK) return rc;
  AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                 H_kv, head_dim, max_blocks_per_seq, block_size);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  cudaError_t e = launch_append_fp8(a, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PAGED_ATTN_OK : cuda_fail(e);
}

int paged_attn_append_decode_fp8(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                 void* out, const int32_t* block_tables, const int32_t* seq_lens,
                                 int num_seqs, int H_q, int H_kv, int head_dim,
                                 int max_blocks_per_seq, int block_size, float scale,
                                 void* stream) {
  int rc = fp8_checks(q, k_cache, v_cache, k_scale, v_scale, out, block_tables, seq_lens,
                      num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  if (!aligned16(k_new) || !aligned16(v_new)) return PAGED_ATTN_ERR_POINTER;
  int dev = 0;
  DeviceInfo di;
  if ((rc = device_info(&di, &dev)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = cached_plan(num_seqs, H_q, H_kv, head_dim, block_size, dev, di, &pl, true)) !=
      PAGED_ATTN_OK)
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.k_scale = k_scale;
  o.v_scale = v_scale;
  apply_checks(&o);
  if ((rc = owned_workspace(pl.ws_bytes, st, &o.ws)) != PAGED_ATTN_OK) return rc;
  // As for bf16 caches: fused (each piece's last page quantized and patched in
  // shared memory, then stored) unless CTAs average kAppendApartPieces or more
  // pieces, when the append runs as its own launch and the decode after it is
  // a plain launch.
  // The fused form is compiled for head_dim 128 only (at 256 its code would cost
  // the page loop a register spill).
  if (head_dim != 128 ||
      (long long)num_seqs * H_kv >= (long long)kAppendApartPieces * pl.grid) {
    AppendParams a = append_params(k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                   num_seqs, H_kv, head_dim, max_blocks_per_seq, block_size);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = launch_append_fp8(a, di.sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    o.early = false;  // the decode reads the rows just appended
    return run(pl, o, st);
  }
  o.early = early_requested();
  o.k_new = k_new;
  o.v_new = v_new;
  return run(pl, o, st);
}

size_t paged_attn_workspace_bytes(int num_seqs, int H_q, int H_kv, int head_dim,
                                  int max_blocks_per_seq, int block_size) {
  if (validate_sizes(num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size) !=
      PAGED_ATTN_OK)
    return 0;
  int dev = 0;
  DeviceInfo di;
  if (device_info(&di, &dev) != PAGED_ATTN_OK) return 0;
  Plan pl;
  if (cached_plan(num_seqs, H_q, H_kv, head_dim, block_size, dev, di, &pl) != PAGED_ATTN_OK)
    return 0;
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
  int dev = 0;
  DeviceInfo di;
  if ((rc = device_info(&di, &dev)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = cached_plan(num_seqs, H_q, H_kv, head_dim, block_size, dev, di, &pl)) !=
      PAGED_ATTN_OK)
    return rc;
  if (workspace_bytes < pl.ws_bytes) return PAGED_ATTN_ERR_WORKSPACE;
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.ws = workspace;
  o.early = early_requested();
  apply_checks(&o);
  return run(pl, o, static_cast<cudaStream_t>(stream));
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
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.num_blocks = num_blocks;
  o.status = d_status;
  o.early = early_requested();
  return plan_and_run(o, head_dim, block_size, false, false, 0, 0,
                      static_cast<cudaStream_t>(stream));
}

int paged_attn_decode_static(const void* q, const void* k_cache, const void* v_cache, void* out,
                             const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                             int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                             int block_size, float scale, void* stream) {
  int rc = common_checks(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                         head_dim, max_blocks_per_seq, block_size, scale);
  if (rc != PAGED_ATTN_OK || num_seqs == 0) return rc;
  int dev = 0;
  DeviceInfo di;
  if ((rc = device_info(&di, &dev)) != PAGED_ATTN_OK) return rc;
  Plan pl;
  if ((rc = cached_plan(num_seqs, H_q, H_kv, head_dim, block_size, dev, di, &pl)) !=
      PAGED_ATTN_OK)
    return rc;
  if (pl.ws_bytes > kStaticScratchBytes) return PAGED_ATTN_ERR_STATIC_SCRATCH;
  void* ws = nullptr;
  if ((rc = static_scratch_address(&ws)) != PAGED_ATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left; the status word and the
  // combine counters must start at zero.  The memset is a plain stream
  // operation ahead of the launch, which then waits for it before touching the
  // array (the early prologue only reads the caller's tables and caches early).
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.off_partials, st);
  if (e != cudaSuccess) return cuda_fail(e);
  Operands o = operands(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                        max_blocks_per_seq, scale);
  o.ws = ws;
  o.early = early_requested();
  apply_checks(&o);
  return run(pl, o, st);
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

int paged_attn_set_checks(long long num_blocks, int32_t* d_status) {
  if (num_blocks <= 0 && d_status == nullptr) {
    g_check_blocks = 0;
    g_check_status = nullptr;
    return PAGED_ATTN_OK;
  }
  if (num_blocks <= 0 || num_blocks > 0x7fffffffLL) return PAGED_ATTN_ERR_SIZES;
  if (d_status == nullptr || (reinterpret_cast<uintptr_t>(d_status) & 3) != 0)
    return PAGED_ATTN_ERR_POINTER;
  g_check_blocks = num_blocks;
  g_check_status = d_status;
  return PAGED_ATTN_OK;
}

int paged_attn_reset_workspace(void* stream) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != PAGED_ATTN_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  const OwnedWorkspace& w = g_ws[dev];
  if (w.ptr == nullptr) return PAGED_ATTN_OK;
  cudaError_t e = cudaMemsetAsync(w.ptr, 0, w.bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PAGED_ATTN_OK : cuda_fail(e);
}

int paged_attn_last_cuda_error(void) { return g_last_cuda_error; }

int paged_attn_version(void) { return 200; }

#ifdef PAGED_ATTN_WAIT_TEST
// Test build only (not in include/paged_attn.h): the next decode launches of
// this thread leave unit `skip_unit` of CTA 0's range without a copy (-1: off)
// and, with skip_publish != 0, make every combiner wait for one more published
// part than exists, so the bounded waits run out.
__attribute__((visibility("default"))) int paged_attn_test_set_wait_faults(int skip_unit,
                                                                           int skip_publish) {
  g_test_skip_unit = skip_unit;
  g_test_skip_publish = skip_publish;
  return PAGED_ATTN_OK;
}
#endif

}  // extern "C"
