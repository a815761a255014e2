// Split-KV paged GQA decode attention for GB300 (sm_103a).
//
// What it computes is the operation of include/paged_attn.h ("Paged Attention
// Kernel Architecture for BI-V100", section 1; paging layout and head map of
// the RL.cu "Add Cuda Kernel" tutorial's paged decode).  How:
//
//  * Work split (section 6 of the BI-V100 design splits each sequence into
//    fixed 512-token partitions; here the split is re-derived for ragged
//    batches): the units of work are pages (s, g, p) -- one physical block of
//    one KV head.  Flattened in (s, g, p) order they are cut into C
//    contiguous ranges, one per persistent CTA (two CTAs per SM, C reduced so
//    each CTA gets at least kMinPagesPerCta pages), of equal weight: a page
//    weighs one and each (s, g) piece adds a fixed weight for its end phase
//    (first_unit).  CTAs stream about the same number of bytes whatever the
//    length mix, and a range crossing (s, g) boundaries simply produces one
//    partial softmax state per piece.
//
//  * Data movement: a producer warp walks the range, reads the block table
//    and issues TMA tiled loads (cp.async.bulk.tensor.4d) into a ring of
//    shared-memory stages, several lanes issuing at once.  One load brings a
//    whole page of one KV head (block_size x head_dim, contiguous in HBM):
//    the 4-D tensor map views a row as two-or-more 64-column halves so the
//    page lands as [half][row][128 B] with the 128-byte swizzle; each stage
//    holds the K page and the V page and completes on one mbarrier.
//
//  * Math (tensor cores, bf16 m16n8k16, fp32 accumulate), with the page's
//    tokens as the M dimension and the GQA group as N (8 heads per n-tile):
//    S^T = K Q^T (K read with ldmatrix from the swizzled tile, Q^T with
//    ldmatrix from the piece's query tile in shared memory), online softmax
//    in fp32 on the accumulator fragments (BI-V100 design, section 2, Level
//    1: running max, exp-sum and weighted V; the max is raised only when a
//    page passes it by kLazyMaxLog2), P^T turned into the B operand
//    with movmatrix, then O^T += V^T P^T (V read with ldmatrix.trans).  Every
//    K/V byte leaves HBM once and feeds all G heads of its group.  The FP8,
//    x-packed and multi-token variants change the operands' loads, the
//    conversions and the query rows, not this structure (see process_fp8,
//    the XP branches and qrow / row_limit).
//
//  * Merge (BI-V100 design, section 2, Levels 2 and 3): at the end of each
//    (s, g) piece the consumer warps merge their states through shared
//    memory.  A piece that is the whole (s, g) is normalised and stored as
//    bf16.  A piece of a split (s, g) is stored as an fp32 partial state; the
//    last CTA to finish a piece of that (s, g) -- found with an atomic counter,
//    so no CTA ever waits for another -- merges all partials in a fixed order
//    and writes the output.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "smem_layout.h"

namespace pagedattn {

constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// Two independent pipelines per SM, except (a) head_dim 256 with more than 8
// query rows, whose accumulators need the whole register file, and (b) bf16
// stages of 16 KB or more (head_dim 256, or 32-token pages): two CTAs could
// hold only one ring slot per consumer warp, which then idles while its next
// page loads; one CTA with two slots a warp and the registers of a whole SM
// streams faster (Qwen-shaped 100K decode 246 -> 237 us, GQA-8 batch 306 -> 303
// us).  FP8 stages are half as large and its consumers need the warps: at
// head_dim 128 with 16-token pages and up to 8 query rows, three CTAs per SM
// (15 warps, 128 registers a thread, no spills; 12-stage rings) decode the
// LLaMA-shaped batch in 31.0 us against 34.2 with two, the ragged 256-sequence
// batch in 320 against 378 us.  (Four CTAs spill and are slower; with
// 32-token pages three are slower, 163 -> 202 us on the GQA-8 batch.)
__host__ __device__ constexpr int ctas_per_sm(int D, bool g16, int BS = 16, bool fp8 = false) {
  return (D >= 256 && g16) || (!fp8 && D * BS * 2 * 2 >= (16 << 10)) ? 1
         : fp8 && D == 128 && BS == 16 && !g16                        ? 3
                                                                      : 2;
}
constexpr int kMaxCtasPerSm = 3;  // the largest ctas_per_sm
constexpr int kMinPagesPerCta = 8;
// Fixed cost of one (sequence, KV head) piece in pages, for the work split.
#ifndef PAGED_ATTN_PIECE_WEIGHT_BF16
#define PAGED_ATTN_PIECE_WEIGHT_BF16 4
#endif
#ifndef PAGED_ATTN_PIECE_WEIGHT_FP8
#define PAGED_ATTN_PIECE_WEIGHT_FP8 4
#endif
// FP8 with three CTAs per SM: a CTA streams a third of an SM, so a piece's
// fixed cost is worth more pages (swept 2-12: 8 best on the LLaMA-shaped batch,
// 30.4 against 31.0 us at 4; 6 best on the ragged 256-sequence batch, 314
// against 323 us at 4 and 317 at 8).
#ifndef PAGED_ATTN_PIECE_WEIGHT_FP8_3CTA
#define PAGED_ATTN_PIECE_WEIGHT_FP8_3CTA 8
#endif
#ifndef PAGED_ATTN_PIECE_WEIGHT_MULTI
#define PAGED_ATTN_PIECE_WEIGHT_MULTI 10
#endif
constexpr int kMaxStages = 16;  // ring depth cap (slot s belongs to consumer warp s % 4)
constexpr int kMaxIssueLanes = 4;   // producer lanes issuing loads at once
constexpr int kConsumerBarrier = 1;
// KV cache formats: bf16 [num_blocks, H_kv, BS, D]; FP8 e4m3 in that layout with
// per-row floats; bf16 x-packed K / D-major V.
constexpr int kKvBf16 = 0;
constexpr int kKvFp8 = 1;
constexpr int kKvXpacked = 2;
// Block tables up to this size are prefetched into L2 at kernel entry.
constexpr size_t kBlockTablePrefetchBytes = size_t(4) << 20;

// Status bits written to the workspace / caller status word.
constexpr int kStatusBadBlock = 1;
constexpr int kStatusBadLength = 2;
constexpr int kStatusTimeout = 4;
constexpr int kStatusConfig = 8;

// Polls before the combiner gives up waiting for the other parts of a split to
// be published (each poll sleeps ~64 ns: about 0.3 s in all).  The test build
// of the library uses a few thousand, so that a test can make it run out fast.
#ifndef PAGED_ATTN_PUBLISH_POLLS
#define PAGED_ATTN_PUBLISH_POLLS (1u << 22)
#endif
constexpr uint32_t kPublishPolls = PAGED_ATTN_PUBLISH_POLLS;

// Lazy rescaling of the online softmax (log2 domain): a warp's running max
// is raised only when some score of a page exceeds it by more than this, so
// most pages skip the cross-lane max and the rescale of the accumulators.
// Weights are then up to 2^4 instead of 1; the result is the same softmax
// (every state is taken against its own max, and merges rescale by those).
// For FP8 caches the f16 weight times the V row float stays finite while
// that float is below 65504 / 16 = 4094.
constexpr float kLazyMaxLog2 = 4.f;

struct DecodeParams {
  const __nv_bfloat16* q;       // [num_seqs, H_q, D]
  __nv_bfloat16* out;           // [num_seqs, H_q, D]
  const int32_t* block_tables;  // [num_seqs, maxb]
  const int32_t* seq_lens;      // [num_seqs]
  int num_seqs;
  int H_q;
  int H_kv;
  int G;
  int maxb;
  int stages;
  float scale_log2;     // softmax scale * log2(e)
  int32_t* status;      // status bits (device int32)
  int32_t* counters;    // [gridDim.x], zero between calls (one per split piece's first CTA)
  float* partials;      // [gridDim.x * 2][G][D + 4]
  long long num_blocks; // > 0: checked mode (validate block ids against it)
  // Fused cache append (null k_new: none): the new token's rows, written into
  // the caches before the pages holding them are read.
  const __nv_bfloat16* k_new;  // [num_seqs, H_kv, D]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache;      // [num_blocks, H_kv, BS, D]
  __nv_bfloat16* v_cache;
  // FP8 caches: one dequant float per (block, KV head, slot) for K and for V
  const float* k_scale;        // [num_blocks, H_kv, BS]
  const float* v_scale;
  // Multi-token decode (null qo_indptr: one query token per sequence).  Sequence
  // s owns rows qo_indptr[s] .. qo_indptr[s+1] - 1 of q and out ([rows, H_q, D]):
  // its last q_len tokens, query i seeing the tokens t <= seq_len - q_len + i.
  // The q_len * G query rows of one KV head (token-major: row r is query r / G,
  // head r % G of the group) are split into `chunks` pieces of `rows` rows.
  const int32_t* qo_indptr;
  int rows;
  int chunks;
  int total_q;  // rows of q and out (offsets outside [0, total_q) are never touched)
  int causal;   // multi-token decode: 1 = query i sees t <= seq_len - q_len + i; 0 = all t < seq_len
  // Early prologue: the caller guarantees that the work still running ahead of
  // this launch in the stream writes none of the caches (and their row floats),
  // block tables, lengths or query offsets.  The producer then reads them and
  // starts its tensor copies without waiting for that work; the consumers (the
  // only ones to read q or the new rows, or to write out or the workspace)
  // still wait for it.
  int early;
#ifdef PAGED_ATTN_WAIT_TEST
  // Test build only: CTA 0 arms the ring slot of its unit `test_skip_unit` but
  // issues no copy into it, so the consumer's bounded wait for that page runs
  // out; CTA `test_skip_publish` never publishes its partial state, so the
  // combiner's bounded wait for it runs out.  -1: off.
  int test_skip_unit;
  int test_skip_publish;
#endif
};

// a / b for 0 <= a, 0 < b, in 32-bit arithmetic when both fit (a 64-bit
// division is a long emulated sequence, and these sit ahead of the first copy).
__device__ __forceinline__ long long div_nonneg(long long a, long long b) {
  if (((unsigned long long)a | (unsigned long long)b) <= 0xffffffffull)
    return (long long)((unsigned int)a / (unsigned int)b);
  return a / b;
}

// Position of one unit (page of one KV head) in the flattened (s, g, p) order.
struct Walker {
  int s, g, p, n;  // sequence, KV head, page within the sequence, pages of the sequence

  __device__ void start(long long u, const int* prefix, int N, int H_kv) {
    int lo = 0, hi = N - 1;  // largest s with prefix[s] * H_kv <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)prefix[mid] * H_kv <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    s = lo;
    n = prefix[s + 1] - prefix[s];
    const long long off = u - (long long)prefix[s] * H_kv;
    g = (int)div_nonneg(off, n);
    p = (int)(off - (long long)g * n);
  }

  __device__ void next(const int* prefix, int N, int H_kv) {
    if (++p < n) return;
    p = 0;
    if (++g < H_kv) return;
    g = 0;
    do {
      ++s;
    } while (s < N && prefix[s + 1] == prefix[s]);
    n = s < N ? prefix[s + 1] - prefix[s] : 0;
  }

  // k units further on (the target unit must exist); one step per piece crossed.
  __device__ void advance(int k, const int* prefix, int N, int H_kv) {
    p += k;
    while (p >= n) {
      p -= n;
      if (++g == H_kv) {
        g = 0;
        do {
          ++s;
        } while (s < N && prefix[s + 1] == prefix[s]);
        if (s >= N) {
          n = 0;
          p = 0;
          return;
        }
        n = prefix[s + 1] - prefix[s];
      }
    }
  }
};

// The CTA whose range contains unit u, for ranges [floor(c W / C), floor((c+1) W / C)).
__device__ __forceinline__ int cta_of(long long u, long long W, long long C) {
  return (int)div_nonneg((u + 1) * C - 1, W);
}

__device__ __forceinline__ long long range_begin(long long c, long long W, long long C) {
  return div_nonneg(c * W, C);
}

// The work split runs over weighted positions: unit p of piece (sw, g) sits at
// H_kv * wprefix[sw] + g * (n + wgt) + p (n: the pages of walked sequence sw),
// and the wgt positions after a piece's units stand for its fixed cost (the
// merge of the warps' states, the output or partial store, the next query
// group) and belong to no unit.  Returns the first unit at or after position T
// (W, the unit count, past the end; Wt: the weighted total).
__device__ __forceinline__ long long first_unit(long long T, long long W, long long Wt,
                                                const int* prefix, const int* wprefix, int NW,
                                                int H_kv, int wgt) {
  if (T >= Wt) return W;
  int lo = 0, hi = NW - 1;  // largest sw with H_kv * wprefix[sw] <= T: a sequence with pages
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)wprefix[mid] * H_kv <= T)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int n = prefix[lo + 1] - prefix[lo];
  if (n == 0) return (long long)prefix[lo + 1] * H_kv;  // (not reached for T < Wt)
  const long long off = T - (long long)wprefix[lo] * H_kv;
  const long long g = div_nonneg(off, n + wgt), r = off - g * (n + wgt);
  const long long base = (long long)prefix[lo] * H_kv + g * n;
  return r < n ? base + r : base + n;
}

// Fused cache append into an FP8 page held in shared memory: the new token's
// bf16 K and V rows (at `rows`: D values of K, then D of V) are quantized as the
// standalone FP8 append does -- float f = max|x| / 448 (1 for a zero row), byte
// = e4m3(x / f) rounded to nearest even, saturating -- and written into row
// `slot` of the page's K and V tiles (128-byte swizzle) and into that row's
// floats (`scales`: BS K floats, then BS V floats).  One warp; lane l holds the
// values l * D / 32 .. of each row.  Out of line: its registers are spent only
// when a page holds a new token, not in the page loop around it.
template <int D>
__device__ __noinline__ void fp8_patch_row(const uint8_t* rows, uint8_t* st, int page_bytes,
                                           int tile_bytes, int slot, float* scales, int BS,
                                           int lane) {
  constexpr int kE = D / 32;
  const __nv_bfloat16* kr = reinterpret_cast<const __nv_bfloat16*>(rows) + lane * kE;
  const __nv_bfloat16* vr = kr + D;
  float xk[kE], xv[kE], ak = 0.f, av = 0.f;
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    xk[e] = __bfloat162float(kr[e]);
    xv[e] = __bfloat162float(vr[e]);
    ak = fmaxf(ak, fabsf(xk[e]));
    av = fmaxf(av, fabsf(xv[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, o));
    av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
  }
  const float fk = ak > 0.f ? ak / 448.f : 1.f;  // IEEE division (no fast math)
  const float fv = av > 0.f ? av / 448.f : 1.f;
  // byte lane * kE of the row: 16-byte chunk c (128-byte half c / 8, swizzled
  // position c ^ slot % 8 within it), offset o in the chunk
  const int c = (lane * kE) >> 4, o = (lane * kE) & 15;
  const int off = (c >> 3) * tile_bytes + slot * 128 + (((c & 7) ^ (slot & 7)) << 4) + o;
#pragma unroll
  for (int k = 0; k < kE / 4; ++k) {
    uint32_t kw = 0u, vw = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      kw |= (uint32_t)__nv_cvt_float_to_fp8(xk[4 * k + b] / fk, __NV_SATFINITE, __NV_E4M3)
            << (8 * b);
      vw |= (uint32_t)__nv_cvt_float_to_fp8(xv[4 * k + b] / fv, __NV_SATFINITE, __NV_E4M3)
            << (8 * b);
    }
    *reinterpret_cast<uint32_t*>(st + off + 4 * k) = kw;
    *reinterpret_cast<uint32_t*>(st + page_bytes + off + 4 * k) = vw;
  }
  if (lane == 0) {
    scales[slot] = fk;
    scales[BS + slot] = fv;
  }
}

// FP8: the caches hold e4m3 bytes (head_dim 128 or 256) and one float per cache// FP8: the caches hold e4m3 bytes (head_dim 128 or 256) and one float per cache
// row; the products run on f16 tensor cores (e4m3 -> f16 is exact, q is turned
// into f16 once per piece), the K row floats scale the scores and the V row
// floats are folded into the probabilities.
//
// XP (x-packed): bf16 caches with K as [num_blocks, H_kv, D / 8, BS, 8] and V as
// [num_blocks, H_kv, D, BS] ("Paged Attention Kernel Architecture for BI-V100",
// section 3).  A K page lands in shared memory as [D / 8][BS][16 bytes] and a V
// page as [D][BS] (V^T, 32- or 64-byte rows), so both MMA operands come from
// plain ldmatrix with other addresses; everything else is the bf16 path.
//
// MULTI: multi-token decode (DecodeParams::qo_indptr); compiled separately so
// the single-token decode carries none of its row mapping or causal masking.
template <int D, int BS, bool G16, int KV = kKvBf16, bool MULTI = false>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(D, G16, BS, KV == kKvFp8))
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  constexpr bool FP8 = KV == kKvFp8;
  constexpr bool XP = KV == kKvXpacked;
  using L = SmemLayout<D, BS, FP8>;
  static_assert(!FP8 || D >= 128, "FP8 caches need head_dim 128 or 256");
  constexpr int kTileBytes = L::kTileBytes;
  constexpr int kPageBytes = L::kPageBytes;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int kRowStride = L::kRowStride;
  constexpr int kPartialRow = D + 4;  // [M, L, pad, pad, o[0..D)]
  constexpr int kNH = G16 ? 2 : 1;    // n8 tiles of query heads
  constexpr int kDT = D / 16;         // 16-wide tiles of head_dim
  constexpr int kTG = BS / 16;        // 16-token groups per page
  constexpr int kQRows = 8 * kNH;                 // query rows one tile holds
  constexpr int kQTileBytes = kQRows * D * 2;     // = lay.q_tile_bytes()
  constexpr int kQ16Stride = L::kQ16Stride;      // FP8: padded f16 query row
  // the fused append's new rows and block id, after the tile (and its f16 copy)
  constexpr int kAppendOff = kQTileBytes + (FP8 ? kQRows * kQ16Stride : 0);
  constexpr bool kFp8FusedAppend = FP8 && D == 128;  // FP8 caches: fused append compiled in
  constexpr int kQSlotBytes = (kAppendOff + 4 * D + 16 + 127) / 128 * 128;  // = lay.q_slot_bytes()

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr bool multi = MULTI;
  const L lay{p.stages, multi ? p.rows : p.G, p.num_seqs, multi ? p.num_seqs + 1 : 0,
              multi ? p.chunks : 1};
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + lay.bars());
  uint64_t* empty_bar = full_bar + p.stages;
  uint64_t* comb_bar = empty_bar + p.stages;  // the combine's partial-state copies
  float* sm_m = reinterpret_cast<float*>(smem + lay.merge_m());
  float* sm_l = reinterpret_cast<float*>(smem + lay.merge_l());
  int* sm_flag = reinterpret_cast<int*>(smem + lay.flag());
  float* sm_o = reinterpret_cast<float*>(smem + lay.merge_o());
  uint8_t* sm_q = smem + lay.qtile();
  float* sm_scales = reinterpret_cast<float*>(smem + lay.scales());  // FP8: [stages][2][BS]
  int* sm_prefix = reinterpret_cast<int*>(smem + lay.prefix());
  int* sm_wprefix = reinterpret_cast<int*>(smem + lay.wprefix());
  int* sm_len = reinterpret_cast<int*>(smem + lay.lens());
  int* sm_qo = reinterpret_cast<int*>(smem + lay.qo());  // multi: qo_indptr[0..N]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int N = p.num_seqs;
  const int H_kv = p.H_kv;
  const int G = p.G;
  const int R = multi ? p.rows : G;      // query rows of one piece
  const int QC = multi ? p.chunks : 1;   // pieces per (sequence, KV head)
  // Multi-token decode with QC > 1 walks the sequences QC times, pass c for row
  // chunk c of every KV head (chunk-major, so the passes over the same pages
  // run at the same time on different CTAs and the repeated reads hit L2):
  // walked sequence sw = c * N + s.
  const int NW = N * QC;
  const int cap = p.maxb * BS;
  // (a multi-token piece of one 8-row tile and one pass costs what a decode
  // piece costs, and splits as the decode does)
  const int kWgt = FP8 ? (ctas_per_sm(D, G16, BS, true) == 3 ? PAGED_ATTN_PIECE_WEIGHT_FP8_3CTA
                                                             : PAGED_ATTN_PIECE_WEIGHT_FP8)
                 : MULTI && (R > 8 || QC > 1) ? PAGED_ATTN_PIECE_WEIGHT_MULTI
                                              : PAGED_ATTN_PIECE_WEIGHT_BF16;
  // Status bits are written only after the work ahead in the stream has
  // completed: with the early prologue the producer runs before that point,
  // and a caller that zero-fills the status word in that work must not erase
  // what this launch reports.  (A no-op wait once it has returned, and for a
  // launch without the programmatic attribute.)
  auto report = [&](int bits) {
    if (p.early) griddep_wait();
    atomicOr(p.status, bits);
  };

  // ---- 0. Programmatic dependent launch: let the next kernel in the stream be
  // scheduled as this grid's CTAs retire, and wait for the previous kernel
  // (which may write any of the inputs) to complete before touching global
  // memory; with the early prologue only the consumers wait (below).  Both are
  // no-ops for a launch without the programmatic attribute.
  griddep_launch_dependents();
  // Start the cold fetches that only depend on the arguments: the tensor maps
  // (kernel parameters, safe before the wait; needed by the first tensor copy)
  // and, spread over the grid, the block table (read right after the prefix
  // below), so neither waits behind the lengths.
  if (tid == kThreads - 32) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (!p.early) griddep_wait();
  {
    const size_t bt_bytes = (size_t)N * p.maxb * sizeof(int32_t);
    if (bt_bytes <= kBlockTablePrefetchBytes) {
      const char* bt = reinterpret_cast<const char*>(p.block_tables);
      for (size_t off = ((size_t)blockIdx.x * kThreads + tid) * 128; off < bt_bytes;
           off += (size_t)gridDim.x * kThreads * 128)
        prefetch_l2(bt + off);
    }
  }

  // ---- 1. clamped lengths, the exclusive prefix of pages per sequence and the
  // same prefix with every piece weighted by its fixed cost (first_unit)
  {
    const int per = (N + kThreads - 1) / kThreads;
    const int s0 = tid * per;
    const int s1 = min(N, s0 + per);
    int local = 0, wlocal = 0;
    for (int s = s0; s < s1; ++s) {
      int len = __ldg(p.seq_lens + s);
      if (len < 0 || len > cap) {
        if (p.num_blocks > 0 && blockIdx.x == 0) report(kStatusBadLength);
        len = min(max(len, 0), cap);
      }
      sm_len[s] = len;
      const int pages = (len + BS - 1) / BS;
      local += pages;
      wlocal += pages + (pages > 0 ? kWgt : 0);
    }
    int incl = local, wincl = wlocal;  // block-wide exclusive scans of both
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      const int wv = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) {
        incl += v;
        wincl += wv;
      }
    }
    __shared__ int warp_tot[kThreads / 32], warp_wtot[kThreads / 32];
    if (lane == 31) {
      warp_tot[warp] = incl;
      warp_wtot[warp] = wincl;
    }
    __syncthreads();
    int base = 0, wbase = 0;
    for (int w = 0; w < warp; ++w) {
      base += warp_tot[w];
      wbase += warp_wtot[w];
    }
    int run = base + incl - local, wrun = wbase + wincl - wlocal;
    for (int s = s0; s < s1; ++s) {
      sm_prefix[s] = run;
      sm_wprefix[s] = wrun;
      const int pages = (sm_len[s] + BS - 1) / BS;
      run += pages;
      wrun += pages + (pages > 0 ? kWgt : 0);
    }
    if (tid == kThreads - 1) {
      sm_prefix[N] = base + incl;
      sm_wprefix[N] = wbase + wincl;
    }
    if (multi) {
      for (int s = tid; s <= N; s += kThreads) sm_qo[s] = __ldg(p.qo_indptr + s);
    }
    __syncthreads();
    if (multi && QC > 1) {  // prefixes of the later passes: offset by c * (all pages)
      const int P = sm_prefix[N], WP = sm_wprefix[N];
      for (int i = tid; i < (QC - 1) * N; i += kThreads) {
        const int c = 1 + i / N;
        const int sq = i - (c - 1) * N;
        sm_prefix[c * N + sq] = c * P + sm_prefix[sq];
        sm_wprefix[c * N + sq] = c * WP + sm_wprefix[sq];
      }
      if (tid == 0) {
        sm_prefix[NW] = QC * P;
        sm_wprefix[NW] = QC * WP;
      }
      __syncthreads();
    }
    if (multi && blockIdx.x == 0) {
      // rows a sequence cannot hold (q_len < 0, or more than the pieces carry) are
      // reported; they are never read or written
      for (int s = tid; s < N; s += kThreads) {
        const int ql = sm_qo[s + 1] - sm_qo[s];
        if (ql < 0 || (long long)ql * G > (long long)R * QC) report(kStatusBadLength);
      }
    }
  }

  // ---- 2. empty sequences get zero rows: sequence s by CTA s mod `ctas`,
  // threads t0, t0 + nt, ... of it
  auto zero_empty = [&](long long ctas, int t0, int nt) {
    for (long long s = blockIdx.x; s < N; s += ctas) {
      if (sm_len[s] != 0) continue;
      const int r0 = multi ? min(max(sm_qo[s], 0), p.total_q) : (int)s;
      const int nr = multi ? max(0, min(min(sm_qo[s + 1] - sm_qo[s], R * QC / G), p.total_q - r0))
                           : 1;
      uint32_t* o32 = reinterpret_cast<uint32_t*>(p.out + (size_t)r0 * p.H_q * D);
      for (int i = t0; i < nr * p.H_q * D / 2; i += nt) o32[i] = 0u;
    }
  };

  const long long W = (long long)sm_prefix[NW] * H_kv;
  if (W == 0) {  // nothing to stream: every CTA zeroes its share and leaves
    if (p.early) griddep_wait();
    zero_empty(gridDim.x, tid, kThreads);
    return;
  }
  if (p.stages < kConsumerWarps) {  // the host plan never launches fewer
    if (tid == 0) report(kStatusConfig);
    return;
  }
  const long long C =
      min((long long)gridDim.x, max(1LL, (W + kMinPagesPerCta - 1) / kMinPagesPerCta));
  if ((long long)blockIdx.x >= C) return;
  // (with the early prologue the consumers zero them once they have waited)
  if (!p.early) zero_empty(C, tid, kThreads);
  // CTA c takes the units at weighted positions [c Wt / C, (c + 1) Wt / C): a
  // CTA crossing many short pieces gets fewer pages.  An interval that falls
  // inside the gap after a piece (possible only for tiny batches) holds no
  // units; that CTA is never part of a split, since the CTAs of a split piece
  // are those whose intervals meet the piece's (gap-free) unit positions.
  const long long Wt = (long long)sm_wprefix[NW] * H_kv;
  auto unit_at = [&](long long T) {
    return first_unit(T, W, Wt, sm_prefix, sm_wprefix, NW, H_kv, kWgt);
  };
  const long long u0 = unit_at(range_begin(blockIdx.x, Wt, C));
  const long long u1 = unit_at(range_begin(blockIdx.x + 1, Wt, C));
  if (u0 >= u1) {
    if (p.early) {  // its share of the empty sequences is still to be zeroed
      griddep_wait();
      zero_empty(C, tid, kThreads);
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(comb_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // =================================================================== producer
    const uint64_t policy = l2_evict_first_policy();
    // Lanes issue loads for consecutive units together; never more lanes than
    // stages, so the lanes of one wave always wait on distinct slots.
    const int issue_lanes = min(kMaxIssueLanes, p.stages);
    Walker wk;
    if (u0 + lane < u1) wk.start(u0 + lane, sm_prefix, NW, H_kv);
    auto fetch = [&](long long u) -> int2 {
      // physical block and KV head of this lane's unit (block -1 past the range)
      if (u >= u1) return make_int2(-1, 0);
      const int sq = multi && QC > 1 ? wk.s % N : wk.s;  // the walked sequence's sequence
      int pb = __ldg(p.block_tables + (size_t)sq * p.maxb + wk.p);
      if (p.num_blocks > 0 && (pb < 0 || (long long)pb >= p.num_blocks))
        report(kStatusBadBlock);  // the TMA bounds check reads it as zeros
      return make_int2(pb, wk.g);
    };
    int2 cur = fetch(u0 + lane);
    bool abort = false;
    long long issued_end = u1 - u0;  // units [0, issued_end) were all issued
    long long my_extra = -1;         // a unit past issued_end this lane issued
    for (long long ub = u0; ub < u1 && !abort; ub += 32) {
      // advance this lane's walker to its unit of the next batch and start that load
      int2 nxt = make_int2(-1, 0);
      if (ub + 32 + lane < u1) {
        wk.advance(32, sm_prefix, NW, H_kv);
        nxt = fetch(ub + 32 + lane);
      }
      const int cnt = (int)min(32LL, u1 - ub);
      for (int j0 = 0; j0 < cnt && !abort; j0 += issue_lanes) {
        const int j = j0 + (lane < issue_lanes ? lane : 0);
        const int pb = __shfl_sync(0xffffffffu, cur.x, j);
        const int g = __shfl_sync(0xffffffffu, cur.y, j);
        bool bad = false, issued = false;
        const long long i = ub - u0 + j;  // unit index within this CTA
        if (lane < issue_lanes && j0 + lane < cnt) {
          const int stage = (int)(i % p.stages);
          const uint32_t phase = (uint32_t)((i / p.stages) & 1);
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u)) {
            report(kStatusTimeout);
            bad = true;
          }
#ifdef PAGED_ATTN_WAIT_TEST
          else if (blockIdx.x == 0 && i == p.test_skip_unit) {
            // the slot is neither armed nor filled: its consumer's wait runs out
          }
#endif
          else {
            issued = true;
            uint8_t* st = smem + stage * kStageBytes;
            if constexpr (FP8) {
              // The page's K and V row floats (64 or 128 bytes each) come with
              // 16-byte cp.async, not as two more bulk copies: with 2 KB pages the
              // tensor-copy engine's operations per byte, not the bytes, set the
              // pace (LLaMA-shaped batch 37.0 -> 33.2 us, ragged batch 454 -> 410).
              // The copies complete on the stage's barrier (cp.async.mbarrier.arrive
              // raises its pending count now, before the arrive below, and lowers it
              // when they land).  A block outside a checked pool reads block 0's
              // floats: its rows are zero-filled by the tensor copy anyway.
              const long long b =
                  pb < 0 || (p.num_blocks > 0 && (long long)pb >= p.num_blocks) ? 0 : pb;
              const size_t row = ((size_t)b * H_kv + g) * BS;
              float* sc = sm_scales + (size_t)stage * 2 * BS;
#pragma unroll
              for (int c = 0; c < BS / 4; ++c) {
                cp_async_16(sc + 4 * c, p.k_scale + row + 4 * c, 16);
                cp_async_16(sc + BS + 4 * c, p.v_scale + row + 4 * c, 16);
              }
              cp_async_mbar_arrive(&full_bar[stage]);
            }
            mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
            if constexpr (XP) {
              // a page of one KV head is contiguous in both x-packed caches: K
              // (and V of 16-token pages) come as one bulk copy each; V of 32-token
              // pages through the tensor map, for the 64-byte swizzle (unswizzled
              // 64-byte rows would cost 4-way bank conflicts in the V reads)
              // (a block id outside a checked pool, or negative, reads block 0:
              // a bulk copy has no bounds check of its own)
              const long long b =
                  pb < 0 || (p.num_blocks > 0 && (long long)pb >= p.num_blocks) ? 0 : pb;
              const size_t off = ((size_t)b * H_kv + g) * (size_t)(D * BS);
              bulk_load(st, p.k_cache + off, kPageBytes, &full_bar[stage]);
              if constexpr (BS == 16)
                bulk_load(st + kPageBytes, p.v_cache + off, kPageBytes, &full_bar[stage]);
              else
                tma_load_4d(st + kPageBytes, &tm_v, &full_bar[stage], 0, 0, g, pb, policy);
            } else {
              tma_load_4d(st, &tm_k, &full_bar[stage], 0, g * BS, 0, pb, policy);
              tma_load_4d(st + kPageBytes, &tm_v, &full_bar[stage], 0, g * BS, 0, pb, policy);
            }
          }
        }
        abort = __any_sync(0xffffffffu, bad);
        if (abort) {  // a wait ran out: this wave is the last
          issued_end = ub - u0 + j0;
          if (issued) my_extra = i;
        }
      }
      cur = nxt;
    }
    // Drain: no copy issued by this CTA may still be in flight when it exits.
    // A unit before issued_end - stages was released by its consumer (its slot
    // was reused only after that); the last `stages` units before issued_end
    // were issued, and so were the units of the wave that ran out whose lanes
    // got their slot.  Every wait is bounded.
    if (lane == 0) {
      for (long long i = issued_end > p.stages ? issued_end - p.stages : 0; i < issued_end; ++i) {
#ifdef PAGED_ATTN_WAIT_TEST
        if (blockIdx.x == 0 && i == p.test_skip_unit) continue;  // never issued
#endif
        if (!mbar_wait(&full_bar[i % p.stages], (uint32_t)((i / p.stages) & 1))) {
          report(kStatusTimeout);
          break;
        }
      }
    }
    if (my_extra >= 0 &&
        !mbar_wait(&full_bar[my_extra % p.stages], (uint32_t)((my_extra / p.stages) & 1)))
      report(kStatusTimeout);
    return;
  }

  // ===================================================================== consumers
  // Fragment ownership (m16n8k16): lane holds tokens / head_dim rows lane/4 and
  // lane/4 + 8, and query heads 8 * nh + 2 * (lane % 4) + {0, 1}.
  const int quad = lane & 3;
  const int row = lane >> 2;
  const int ctid = tid;  // 0 .. kConsumerThreads-1
  bool abort = false;    // this warp gave up waiting for a page (status reports it)
  int first_old = -1;    // thread 0: counter value its first piece's arrival saw
  if (p.early) {  // the producer went ahead; q, out and the workspace wait for the previous work
    griddep_wait();
    zero_empty(C, ctid, kConsumerThreads);
  }

  float o_acc[kDT][kNH][4];   // O^T accumulators
  float m_run[kNH][2];        // running max per owned head (log2 domain)
  float l_run[kNH][2];        // running sum per owned head (this lane's tokens)

  // The query group of a piece lives in one of kQSlots shared tiles
  // [16 heads][D] (16-byte chunk c of head h at c ^ (h % 8) within each 128
  // bytes; heads >= G are zero) and is fetched kQSlots - 1 pieces ahead with
  // cp.async, one commit group per piece (an empty group past the range's last
  // piece, so that the group count stays exact).
  // With the fused cache append the slot also receives the piece's new K and V
  // rows and the block id of its last page, so the warp that patches that page
  // finds them in shared memory.
  // Row of q / out ([rows, H_q, D] viewed as rows of D) that row r of piece
  // (sw, g) stands for, or -1 for a padding row (never stored): walked
  // sequence sw = c * N + s holds row chunk c of sequence s.
  auto qrow = [&](int sw, int g, int r) -> long long {
    if (!multi) return r < G ? (long long)sw * p.H_q + (long long)g * G + r : -1;
    const int c = sw / N;
    const int s = sw - c * N;
    const int rr = c * R + r;  // row within the KV head's q_len * G rows
    const int i = rr / G;
    const long long t = (long long)sm_qo[s] + i;  // the query's row of q / out
    if (r >= R || i >= sm_qo[s + 1] - sm_qo[s] || t < 0 || t >= p.total_q) return -1;
    return t * p.H_q + (long long)g * G + (rr - i * G);
  };
  // Last token row r of piece (sw, g) attends (causal in multi-token decode).
  auto row_limit = [&](int sw, int g, int r) -> int {
    if (!multi) return 0x7fffffff;
    const int c = sw / N;
    const int s = sw - c * N;
    const int i = (c * R + r) / G;
    const int ql = sm_qo[s + 1] - sm_qo[s];
    // padding rows, and every row without the causal mask: no limit
    return i < ql && p.causal ? sm_len[s] - ql + i : 0x7fffffff;
  };
  auto prefetch_q = [&](int buf, int s, int g) {
    uint8_t* tile = sm_q + buf * kQSlotBytes;
    for (int i = ctid; i < kQRows * (D / 8); i += kConsumerThreads) {
      const int h = i / (D / 8);
      const int c = i - h * (D / 8);
      const int pc = (c & ~7) | ((c & 7) ^ (h & 7));
      const long long qr = qrow(s, g, h);
      cp_async_16(tile + h * (D * 2) + pc * 16,
                  qr >= 0 ? static_cast<const void*>(p.q + qr * D + c * 8)
                          : static_cast<const void*>(p.q),
                  qr >= 0 ? 16 : 0);
    }
    if (!multi && !XP && (!FP8 || kFp8FusedAppend) && p.k_new != nullptr) {
      const size_t row = ((size_t)s * H_kv + g) * D;
      for (int i = ctid; i < D / 4; i += kConsumerThreads) {  // K then V, 16 bytes each
        const bool is_v = i >= D / 8;
        const int c = is_v ? i - D / 8 : i;
        cp_async_16(tile + kAppendOff + (is_v ? 2 * D : 0) + c * 16,
                    (is_v ? p.v_new : p.k_new) + row + c * 8, 16);
      }
      if (ctid == kConsumerThreads - 1) {
        const int last_page = sm_prefix[s + 1] - sm_prefix[s] - 1;
        cp_async_4(tile + kAppendOff + 4 * D, p.block_tables + (size_t)s * p.maxb + last_page);
      }
    }
    cp_async_commit();
  };
  // FP8: the slot's bf16 query rows (swizzled, as prefetched) -> f16 rows in
  // natural order, padded (kQ16Stride) so the page loop's 8-byte reads of four
  // rows x four lanes fall in distinct banks.  Each thread converts the 16-byte
  // chunks it copied itself (the same index walk as prefetch_q), which its own
  // cp.async.wait_all has made visible to it, so no barrier is needed between
  // the copies landing and the conversion; the barrier after it publishes the
  // f16 rows.
  auto convert_own_q = [&](int buf) {
    const uint8_t* tile = sm_q + buf * kQSlotBytes;
    uint8_t* q16 = sm_q + buf * kQSlotBytes + kQTileBytes;
    for (int i = ctid; i < kQRows * (D / 8); i += kConsumerThreads) {
      const int h = i / (D / 8);
      const int c = i - h * (D / 8);
      const int pc = (c & ~7) | ((c & 7) ^ (h & 7));
      const uint4 v = *reinterpret_cast<const uint4*>(tile + h * (D * 2) + pc * 16);
      uint4 o;
      o.x = pack_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x));
      o.y = pack_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
      o.z = pack_f16x2(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z));
      o.w = pack_f16x2(bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
      *reinterpret_cast<uint4*>(q16 + h * kQ16Stride + c * 16) = o;
    }
  };
  int lim[kNH][2];  // last token each of this lane's query columns may see
  auto set_limits = [&](int s, int gv) {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) lim[nh][e] = row_limit(s, gv, 8 * nh + 2 * quad + e);
  };
  auto reset = [&]() {
#pragma unroll
    for (int dt = 0; dt < kDT; ++dt)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_acc[dt][nh][e] = 0.f;
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[nh][e] = -INFINITY;
        l_run[nh][e] = 0.f;
      }
  };

  // One page: S^T = K Q^T, online softmax, O^T += V^T P^T.
  // `tb`: the page's first token; `lim`: the last token each of the lane's
  // query columns may see (causal multi-token decode; the maximum int otherwise).
  auto process_page = [&](const uint8_t* kt, const uint8_t* vt, const uint8_t* qtile,
                          int valid, int tb, const int (&lim)[kNH][2]) {
    const uint32_t kbase = smem_addr(kt);
    const uint32_t vbase = smem_addr(vt);
    const uint32_t qbase = smem_addr(qtile);
    const int li = lane >> 3;  // which 8x8 matrix this lane addresses in ldmatrix.x4
    // Two accumulator sets (even / odd 16-column steps) halve the dependent MMA chain.
    float s_acc[kTG][kNH][4], s_odd[kTG][kNH][4];
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) s_acc[tg][nh][e] = s_odd[tg][nh][e] = 0.f;

    // ---- S^T = K Q^T: A operand = 16 tokens x 16 columns of the swizzled K tile,
    //      B operand Q^T from the query tile
#pragma unroll
    for (int kq = 0; kq < kDT / 2; ++kq) {
      uint32_t qf[2][kNH][2];  // B fragments for column steps 2kq, 2kq+1
      {
        const int chunk = 4 * kq + li;
        const int pc = (chunk & ~7) | ((chunk & 7) ^ (lane & 7));
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh)
          ldmatrix_x4(qbase + (uint32_t)((8 * nh + (lane & 7)) * (D * 2) + pc * 16),
                      qf[0][nh][0], qf[0][nh][1], qf[1][nh][0], qf[1][nh][1]);
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int kk = 2 * kq + x;
        const int chunk = 2 * kk + (li >> 1);
        const uint32_t coff =
            (uint32_t)((chunk >> 3) * kTileBytes + (((chunk & 7) ^ (lane & 7)) << 4));
#pragma unroll
        for (int tg = 0; tg < kTG; ++tg) {
          const int tok = 16 * tg + (lane & 7) + ((li & 1) << 3);
          uint32_t a0, a1, a2, a3;
          if constexpr (XP)  // [D / 8][BS][8]: 16-byte rows, consecutive tokens adjacent
            ldmatrix_x4(kbase + (uint32_t)((chunk * BS + tok) * 16), a0, a1, a2, a3);
          else
            ldmatrix_x4(kbase + coff + (uint32_t)(tok * 128), a0, a1, a2, a3);
#pragma unroll
          for (int nh = 0; nh < kNH; ++nh)
            mma_bf16_16816(x ? s_odd[tg][nh] : s_acc[tg][nh], a0, a1, a2, a3, qf[x][nh][0],
                           qf[x][nh][1]);
        }
      }
    }
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) s_acc[tg][nh][e] += s_odd[tg][nh][e];

    // ---- online softmax per head (log2 domain); masked tokens are selected out
    float mx[kNH][2];
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) mx[nh][0] = mx[nh][1] = -INFINITY;
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 16 * tg + row + ((e >> 1) << 3);
          const float x = tok < valid && (!MULTI || tb + tok <= lim[nh][e & 1])
                              ? s_acc[tg][nh][e] * p.scale_log2
                              : -INFINITY;
          s_acc[tg][nh][e] = x;
          mx[nh][e & 1] = fmaxf(mx[nh][e & 1], x);
        }
    float m_sub[kNH][2];
    float alpha[kNH][2];
    // The running max moves only when a score of the page passes it by more
    // than kLazyMaxLog2; otherwise the weights are taken against the old max
    // (at most 2^kLazyMaxLog2) and nothing is rescaled.
    bool grow = false;
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) grow |= mx[nh][e] > m_run[nh][e] + kLazyMaxLog2;
    const bool changed = __any_sync(0xffffffffu, grow);
    if (changed) {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = mx[nh][e];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          const float m_new = fmaxf(m_run[nh][e], v);
          // a column that has seen no token yet (all masked) keeps -inf; subtract 0
          // then, so its weights are exp2(-inf) = 0 instead of NaN
          m_sub[nh][e] = MULTI && m_new == -INFINITY ? 0.f : m_new;
          alpha[nh][e] = fast_exp2(m_run[nh][e] - m_sub[nh][e]);
          m_run[nh][e] = m_new;
        }
    } else {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          m_sub[nh][e] = MULTI && m_run[nh][e] == -INFINITY ? 0.f : m_run[nh][e];
          alpha[nh][e] = 1.f;
        }
    }
    uint32_t pb0[kTG][kNH], pb1[kTG][kNH];  // B operand P^T (tokens 0-7 / 8-15 of a group)
    float psum[kNH][2];
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) psum[nh][0] = psum[nh][1] = 0.f;
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh) {
        const float e0 = fast_exp2(s_acc[tg][nh][0] - m_sub[nh][0]);
        const float e1 = fast_exp2(s_acc[tg][nh][1] - m_sub[nh][1]);
        const float e2 = fast_exp2(s_acc[tg][nh][2] - m_sub[nh][0]);
        const float e3 = fast_exp2(s_acc[tg][nh][3] - m_sub[nh][1]);
        const uint32_t lo = pack_bf16x2(e0, e1);  // tokens row,   heads 2q, 2q+1
        const uint32_t hi = pack_bf16x2(e2, e3);  // tokens row+8, heads 2q, 2q+1
        psum[nh][0] += bf16lo_to_f32(lo) + bf16lo_to_f32(hi);
        psum[nh][1] += bf16hi_to_f32(lo) + bf16hi_to_f32(hi);
        pb0[tg][nh] = movmatrix_trans(lo);  // tokens 2q, 2q+1 of head `row`
        pb1[tg][nh] = movmatrix_trans(hi);
      }
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) l_run[nh][e] = l_run[nh][e] * alpha[nh][e] + psum[nh][e];
    if (changed) {
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt)
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
          for (int e = 0; e < 4; ++e) o_acc[dt][nh][e] *= alpha[nh][e & 1];
    }

    // ---- O^T += V^T P^T: A operand = 16 columns x 16 tokens via transposing ldmatrix
    const bool tail = valid < BS;
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg) {
      uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
      if (tail) {  // rows past the sequence may hold anything: zero them in the fragment
        const int t0 = 16 * tg + 2 * quad;
        mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
        mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
      }
      const int tok = 16 * tg + (lane & 7) + ((li >> 1) << 3);
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt) {
        uint32_t a0, a1, a2, a3;
        if constexpr (XP) {
          // V^T rows d (BS * 2 bytes each), 16-byte chunk j = 8 tokens; 32-token
          // pages carry the 64-byte TMA swizzle (chunk j stored at j ^ bits 7-8 of
          // the row's address), 16-token pages are a plain copy (2-way conflicts)
          const int d = 16 * dt + (lane & 7) + ((li & 1) << 3);
          const int j = 2 * tg + (li >> 1);
          const int sw = BS == 16 ? 0 : (d >> 1) & 3;
          ldmatrix_x4(vbase + (uint32_t)(d * BS * 2 + ((j ^ sw) << 4)), a0, a1, a2, a3);
        } else {
          const int chunk = 2 * dt + (li & 1);
          const uint32_t addr = vbase + (uint32_t)((chunk >> 3) * kTileBytes + tok * 128 +
                                                   (((chunk & 7) ^ (lane & 7)) << 4));
          ldmatrix_x4_trans(addr, a0, a1, a2, a3);
        }
        a0 &= mlo;
        a1 &= mlo;
        a2 &= mhi;
        a3 &= mhi;
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh)
          mma_bf16_16816(o_acc[dt][nh], a0, a1, a2, a3, pb0[tg][nh], pb1[tg][nh]);
      }
    }
  };

  // FP8 tiles.  The unit of work is a group of NT 16-token tiles (one BS = 16
  // page, or the two halves of a BS = 32 page), each tile with its own K / V
  // shared-memory rows, row floats and count of valid tokens.  S^T = K Q^T on f16 tensor cores: one ldmatrix.x4
  // on the e4m3 K tile hands each lane, for two 16-column steps (two 16-byte
  // chunks), the bytes 4q..4q+3 of its token rows r and r + 8; within each
  // chunk the contraction runs in a fixed permuted order (bytes 4q, 4q+1 ->
  // MMA k 2q, 2q+1; 4q+2, 4q+3 -> 2q+8, 2q+9), and the query operand (f16,
  // natural order) is read in the same order: four consecutive f16 of its row.
  // The K row floats scale the scores; the V row floats are folded into the
  // probabilities.  O^T += V^T P^T: ldmatrix.x4.trans on the e4m3 V tile with
  // byte pairs as 16-bit units hands each lane, for the d pair (2r, 2r+1) and
  // tokens (2q, 2q+1), four bytes that one byte permute splits per d; so the
  // accumulator rows r and r + 8 of a 16-column tile are the columns 2r and
  // 2r + 1.  V rows past the sequence were zeroed in shared memory by the
  // caller, so the V operand needs no mask.
  struct Tile8 {
    uint32_t k, v;        // shared-memory address of the tile's first K / V row
    uint32_t ks, vs;      // shared-memory address of its 16 K / V row floats
    int valid;            // tokens of the tile inside the sequence (0..16)
  };
  auto process_fp8 = [&](auto nt, const Tile8* tl, uint32_t q16) {
    constexpr int NT = decltype(nt)::value;
    const int li = lane >> 3;
    float s_acc[NT][kNH][4], s_odd[NT][kNH][4];
#pragma unroll
    for (int tg = 0; tg < NT; ++tg)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) s_acc[tg][nh][e] = s_odd[tg][nh][e] = 0.f;
    const int trow = (lane & 7) + ((li & 1) << 3);  // tile row this lane addresses
#pragma unroll
    for (int kk2 = 0; kk2 < kDT / 2; ++kk2) {
      uint32_t qf[2][kNH][2];
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh) {
          const uint2 b = lds_u32x2(
              q16 + (uint32_t)((8 * nh + row) * kQ16Stride + (16 * (2 * kk2 + x) + 4 * quad) * 2));
          qf[x][nh][0] = b.x;
          qf[x][nh][1] = b.y;
        }
      const int chunk = 2 * kk2 + (li >> 1);
      const uint32_t coff =
          (uint32_t)((chunk >> 3) * kTileBytes + trow * 128 + (((chunk & 7) ^ (trow & 7)) << 4));
#pragma unroll
      for (int tg = 0; tg < NT; ++tg) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(tl[tg].k + coff, r0, r1, r2, r3);
        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
        e4m3x4_to_f16x2x2(r0, a0, a2);
        e4m3x4_to_f16x2x2(r1, a1, a3);
        e4m3x4_to_f16x2x2(r2, c0, c2);
        e4m3x4_to_f16x2x2(r3, c1, c3);
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh) {
          mma_f16_16816(s_acc[tg][nh], a0, a1, a2, a3, qf[0][nh][0], qf[0][nh][1]);
          mma_f16_16816(s_odd[tg][nh], c0, c1, c2, c3, qf[1][nh][0], qf[1][nh][1]);
        }
      }
    }
    // ---- online softmax per head (log2 domain); masked tokens are selected out
    float mx[kNH][2];
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) mx[nh][0] = mx[nh][1] = -INFINITY;
#pragma unroll
    for (int tg = 0; tg < NT; ++tg) {
      const int valid = tl[tg].valid;
      const float k_lo = p.scale_log2 * lds_f32(tl[tg].ks + 4 * row);
      const float k_hi = p.scale_log2 * lds_f32(tl[tg].ks + 4 * (row + 8));
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = row + ((e >> 1) << 3);
          const float sum = s_acc[tg][nh][e] + s_odd[tg][nh][e];
          const float x = tok < valid ? sum * ((e >> 1) ? k_hi : k_lo) : -INFINITY;
          s_acc[tg][nh][e] = x;
          mx[nh][e & 1] = fmaxf(mx[nh][e & 1], x);
        }
    }
    float alpha[kNH][2];
    bool grow = false;  // as in process_page: the max moves only past kLazyMaxLog2
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) grow |= mx[nh][e] > m_run[nh][e] + kLazyMaxLog2;
    const bool changed = __any_sync(0xffffffffu, grow);
    if (changed) {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = mx[nh][e];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          const float m_new = fmaxf(m_run[nh][e], v);
          alpha[nh][e] = fast_exp2(m_run[nh][e] - m_new);
          m_run[nh][e] = m_new;
        }
    } else {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) alpha[nh][e] = 1.f;
    }
    uint32_t pb0[NT][kNH], pb1[NT][kNH];
    float psum[kNH][2];
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) psum[nh][0] = psum[nh][1] = 0.f;
#pragma unroll
    for (int tg = 0; tg < NT; ++tg) {
      const int valid = tl[tg].valid;
      // masked rows may hold NaN floats
      const float v_lo = row < valid ? lds_f32(tl[tg].vs + 4 * row) : 0.f;
      const float v_hi = row + 8 < valid ? lds_f32(tl[tg].vs + 4 * (row + 8)) : 0.f;
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh) {
        const float e0 = fast_exp2(s_acc[tg][nh][0] - m_run[nh][0]);
        const float e1 = fast_exp2(s_acc[tg][nh][1] - m_run[nh][1]);
        const float e2 = fast_exp2(s_acc[tg][nh][2] - m_run[nh][0]);
        const float e3 = fast_exp2(s_acc[tg][nh][3] - m_run[nh][1]);
        psum[nh][0] += e0 + e2;
        psum[nh][1] += e1 + e3;
        pb0[tg][nh] = movmatrix_trans(pack_f16x2(e0 * v_lo, e1 * v_lo));
        pb1[tg][nh] = movmatrix_trans(pack_f16x2(e2 * v_hi, e3 * v_hi));
      }
    }
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) l_run[nh][e] = l_run[nh][e] * alpha[nh][e] + psum[nh][e];
    if (changed) {
#pragma unroll
      for (int dt = 0; dt < kDT; ++dt)
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
          for (int e = 0; e < 4; ++e) o_acc[dt][nh][e] *= alpha[nh][e & 1];
    }
#pragma unroll
    for (int dt2 = 0; dt2 < kDT / 2; ++dt2) {
      const int chunk = 2 * dt2 + (li >> 1);
      const uint32_t coff =
          (uint32_t)((chunk >> 3) * kTileBytes + trow * 128 + (((chunk & 7) ^ (trow & 7)) << 4));
#pragma unroll
      for (int tg = 0; tg < NT; ++tg) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4_trans(tl[tg].v + coff, r0, r1, r2, r3);
        // r0 / r1: tokens 0-7 / 8-15 of chunk 2 dt2; r2 / r3: of chunk 2 dt2 + 1
        const uint32_t x0 = __byte_perm(r0, 0, 0x3120), x1 = __byte_perm(r1, 0, 0x3120);
        const uint32_t x2 = __byte_perm(r2, 0, 0x3120), x3 = __byte_perm(r3, 0, 0x3120);
        // a0 / a1: columns 2r / 2r+1, tokens 2q, 2q+1; a2 / a3: tokens 2q+8, 2q+9
        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
        e4m3x4_to_f16x2x2(x0, a0, a1);
        e4m3x4_to_f16x2x2(x1, a2, a3);
        e4m3x4_to_f16x2x2(x2, c0, c1);
        e4m3x4_to_f16x2x2(x3, c2, c3);
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh) {
          mma_f16_16816(o_acc[2 * dt2][nh], a0, a1, a2, a3, pb0[tg][nh], pb1[tg][nh]);
          mma_f16_16816(o_acc[2 * dt2 + 1][nh], c0, c1, c2, c3, pb0[tg][nh], pb1[tg][nh]);
        }
      }
    }
  };

  // Head-dimension column of accumulator element e of o_acc[dt] held by this lane.
  auto acc_col = [&](int dt, int e) -> int {
    if constexpr (FP8)
      return 16 * dt + 2 * row + (e >> 1);
    else
      return 16 * dt + row + ((e >> 1) << 3);
  };

  // Partial state slot this CTA writes for a split piece beginning at sb: slot 0
  // for its first piece (begun at or before u0), slot 1 for its last.
  auto my_slot = [&](long long sb) -> int { return 2 * (int)blockIdx.x + (sb <= u0 ? 0 : 1); };

  // A split (s, g): the CTAs c_first..c_last hold its pieces; c_first's piece
  // sits in slot_first, every later CTA's in its slot 0 (its first piece).
  struct Split {
    int s, g, c_first, c_last, slot_first;
  };
  auto make_split = [&](int s, int g, long long sb, long long se) -> Split {
    Split x;
    x.s = s;
    x.g = g;
    const long long n = se - sb;
    const long long xs = (long long)sm_wprefix[s] * H_kv + (long long)g * (n + kWgt);
    x.c_first = cta_of(xs, Wt, C);
    x.c_last = cta_of(xs + n - 1, Wt, C);
    // The piece is c_first's first (slot 0) unless the unit before it -- the
    // previous piece's last, kWgt + 1 positions earlier -- is c_first's too.
    const bool first_of_cta = sb == 0 || cta_of(xs - 1 - kWgt, Wt, C) != x.c_first;
    x.slot_first = 2 * x.c_first + (first_of_cta ? 0 : 1);
    return x;
  };

  // The combine (BI-V100 design, section 2, Level 3) run by the last CTA to
  // arrive for a split: the partial states of c_first..c_last are merged in CTA
  // order and the bf16 rows stored.  Partials are brought into the (now idle)
  // pipeline ring with bulk copies, as many per round as the ring holds (the
  // parts of both splits a CTA may combine share rounds), and folded in online
  // by threads owning float4 slices of the output rows.
  constexpr int kSlots = (8 * kNH * (D / 4) + kConsumerThreads - 1) / kConsumerThreads;
  auto fold = [&](const float* parts, int nc, float4 (&acc)[kSlots], float (&m_acc)[kSlots],
                  float (&l_acc)[kSlots]) {
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      const int v = ctid + k * kConsumerThreads;  // float4 index within [R][D/4]
      if (v >= R * (D / 4)) continue;
      const int r = v / (D / 4), d4 = v - r * (D / 4);
      float m_new = m_acc[k];
#pragma unroll 4
      for (int j = 0; j < nc; ++j) m_new = fmaxf(m_new, parts[(j * R + r) * kPartialRow]);
      if (m_new == -INFINITY) continue;
      const float sc = m_acc[k] == -INFINITY ? 0.f : fast_exp2(m_acc[k] - m_new);
      float4 a = make_float4(acc[k].x * sc, acc[k].y * sc, acc[k].z * sc, acc[k].w * sc);
      float l = l_acc[k] * sc;
#pragma unroll 4
      for (int j = 0; j < nc; ++j) {
        const float* prow = parts + (j * R + r) * kPartialRow;
        const float2 ml = *reinterpret_cast<const float2*>(prow);
        const float4 o4 = *reinterpret_cast<const float4*>(prow + 4 + 4 * d4);
        const float wgt = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - m_new);
        a.x += wgt * o4.x;
        a.y += wgt * o4.y;
        a.z += wgt * o4.z;
        a.w += wgt * o4.w;
        l += wgt * ml.y;
      }
      acc[k] = a;
      l_acc[k] = l;
      m_acc[k] = m_new;
    }
  };
  auto store_rows = [&](const Split& x, const float4 (&acc)[kSlots], const float (&l_acc)[kSlots]) {
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      const int v = ctid + k * kConsumerThreads;
      if (v >= R * (D / 4)) continue;
      const int r = v / (D / 4), d4 = v - r * (D / 4);
      const long long qr = qrow(x.s, x.g, r);
      if (qr < 0) continue;
      const float inv = l_acc[k] > 0.f ? 1.f / l_acc[k] : 0.f;  // a row that saw no token: 0
      uint2 packed;
      packed.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
      packed.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
      *reinterpret_cast<uint2*>(p.out + qr * D + 4 * d4) = packed;
    }
  };
  uint32_t comb_phase = 0;
  // x0 (and x1 when njobs == 2), parts in CTA order.  When local_t >= 0, x0's
  // part number local_t (this CTA's) is not read back from the workspace: its
  // merged state already sits in the ring at that place of the first round.
  auto combine = [&](const Split& x0, const Split& x1, int njobs, int local_t) {
    const int part_bytes = R * kPartialRow * 4;
    const int per_round = (p.stages * kStageBytes) / part_bytes;  // >= 3 for ring >= 4 stages
    if (per_round < 1) {
      if (ctid == 0) report(kStatusConfig);
      return;
    }
    const int n0 = x0.c_last - x0.c_first + 1;
    const int total = n0 + (njobs > 1 ? x1.c_last - x1.c_first + 1 : 0);
    float4 acc[kSlots];
    float m_acc[kSlots], l_acc[kSlots];
    auto reset_acc = [&]() {
#pragma unroll
      for (int k = 0; k < kSlots; ++k) {
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        m_acc[k] = -INFINITY;
        l_acc[k] = 0.f;
      }
    };
    reset_acc();
    for (int t0 = 0; t0 < total; t0 += per_round) {
      const int nt = min(per_round, total - t0);
      if (ctid == 0) {
        fence_proxy_async_all();  // earlier accesses of the ring; the acquired partials
        const bool has_local = local_t >= t0 && local_t < t0 + nt;
        mbar_arrive_expect_tx(comb_bar, (uint32_t)((nt - (has_local ? 1 : 0)) * part_bytes));
        for (int t = t0; t < t0 + nt; ++t) {
          if (t == local_t) continue;  // already in place
          const Split& x = t < n0 ? x0 : x1;
          const int c = x.c_first + (t < n0 ? t : t - n0);
          const int slot = c == x.c_first ? x.slot_first : 2 * c;
          bulk_load(smem + (t - t0) * part_bytes, p.partials + (size_t)slot * R * kPartialRow,
                    (uint32_t)part_bytes, comb_bar);
        }
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(comb_bar, comb_phase & 1u));
      ++comb_phase;
      // one verdict for all consumer warps, so they leave (or go on) together
      if (named_barrier_or(kConsumerBarrier, kConsumerThreads, !ok)) {
        if (ctid == 0) report(kStatusTimeout);
        return;
      }
      for (int t = t0; t < t0 + nt;) {
        const int job_end = t < n0 ? n0 : total;
        const int cnt = min(t0 + nt, job_end) - t;
        fold(reinterpret_cast<const float*>(smem + (t - t0) * part_bytes), cnt, acc, m_acc,
             l_acc);
        t += cnt;
        if (t == job_end) {
          store_rows(t == n0 ? x0 : x1, acc, l_acc);
          reset_acc();
        }
      }
      if (t0 + nt < total) {
        __syncwarp();
        named_barrier(kConsumerBarrier, kConsumerThreads);  // the ring may be refilled
      }
    }
  };

  // Merge the four consumer warps' states of a piece through shared memory
  // (BI-V100 design, section 2, Level 2), with one barrier: every warp stores
  // its (m, l) per head and its unscaled o; emit() then combines the four per
  // output element.  When `arrive` is given, thread 0 arrives on that split
  // counter (a relaxed add: nothing is published yet) as soon as every warp is
  // done with the piece's pages; its old value lands in *old.
  auto merge_warps = [&](int* arrive, int* old) {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_run[nh][e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l_run[nh][e] = v;
      }
    if (row == 0) {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 8 * nh + 2 * quad + e;
          sm_m[warp * 16 + h] = m_run[nh][e];
          sm_l[warp * 16 + h] = l_run[nh][e];
        }
    }
#pragma unroll
    for (int dt = 0; dt < kDT; ++dt)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 8 * nh + 2 * quad + (e & 1);
          const int d = acc_col(dt, e);
          if (h < R) sm_o[(warp * R + h) * kRowStride + d] = o_acc[dt][nh][e];
        }
    __syncwarp();
    named_barrier(kConsumerBarrier, kConsumerThreads);
    if (arrive != nullptr && ctid == 0) *old = atomicAdd(arrive, 1);
  };

  // Combine the warps' states and write the piece's merged state: normalised
  // bf16 rows of (s, g) (whole piece), or a partial row set [M, L, -, -, o]
  // at `dst` (a workspace slot, or part 0 of the ring).  Per row: M = max of
  // the warps' m, each warp's weight 2^(m_w - M) (0 for a warp that saw no
  // token), L and o the weighted sums in warp order.
  auto emit = [&](int s, int g, float* dst) {
    for (int i = ctid; i < R * (D / 4); i += kConsumerThreads) {
      const int r = i / (D / 4);
      const int d = 4 * (i - r * (D / 4));
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = sm_m[w * 16 + r];
        const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
        if (mw != -INFINITY) lsum += sm_l[w * 16 + r] * f;
        const float4 v = *reinterpret_cast<const float4*>(sm_o + (w * R + r) * kRowStride + d);
        acc.x += v.x * f;
        acc.y += v.y * f;
        acc.z += v.z * f;
        acc.w += v.w * f;
      }
      if (dst == nullptr) {
        const long long qr = qrow(s, g, r);
        if (qr < 0) continue;
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;  // a row that saw no token: 0
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(p.out + qr * D + d) = packed;
      } else {
        float* prow = dst + r * kPartialRow;
        *reinterpret_cast<float4*>(prow + 4 + d) = acc;
        if (d == 0) *reinterpret_cast<float2*>(prow) = make_float2(M, lsum);
      }
    }
  };

  // Thread 0: waits (bounded) until the published count (high half) of a split
  // counter reaches `want`, with acquire ordering.  Only CTAs that have already
  // arrived are waited for, and they publish without waiting on anyone.
  auto wait_published = [&](const int* word, int want) -> bool {
    for (uint32_t k = 0; k < kPublishPolls; ++k) {
      if ((ld_acquire_gpu(word) >> 16) >= want) return true;
      __nanosleep(64);
    }
    return false;
  };

  // Pieces of this CTA's range in order: (s, g) and where its units begin.
  struct Piece {
    int s, g;
    long long sb;  // first unit of the whole (s, g)
  };
  auto next_piece = [&](Piece pc) -> Piece {
    if (pc.s >= NW) return pc;  // already past the last walked sequence
    const int n = sm_prefix[pc.s + 1] - sm_prefix[pc.s];
    if (++pc.g == H_kv) {
      pc.g = 0;
      do {
        ++pc.s;
      } while (pc.s < NW && sm_prefix[pc.s + 1] == sm_prefix[pc.s]);
    }
    pc.sb = pc.s < NW ? (long long)sm_prefix[pc.s] * H_kv +
                           (long long)pc.g * (sm_prefix[pc.s + 1] - sm_prefix[pc.s])
                     : pc.sb + n;
    return pc;
  };

  Walker wk;
  wk.start(u0, sm_prefix, NW, H_kv);
  // The range's first and last pieces (the only ones that can be split) and
  // their split descriptors, worked out now by thread 0 (off the critical path
  // at the end) and kept in shared memory, not in registers, through the loop.
  Split* const sm_split = reinterpret_cast<Split*>(sm_flag + 4);  // [0] first, [1] last
  int* const sm_split_flags = sm_flag + 4 + 2 * (int)(sizeof(Split) / sizeof(int));
  // The query slots: the current piece's (qbuf) and the next kQSlots - 1
  // pieces' in the slots after it; `ahead` is the next piece to prefetch.
  auto prefetch_or_skip = [&](int buf, const Piece& pc) {
    if (pc.s < NW && pc.sb < u1)
      prefetch_q(buf, pc.s, pc.g);
    else
      cp_async_commit();  // an empty group keeps the count
  };
  int qbuf = 0;
  prefetch_q(0, wk.s, wk.g);
  Piece ahead = next_piece(Piece{wk.s, wk.g, 0});
  if (ctid == 0) {  // while the first query group is in flight
    const long long first_sb = (long long)sm_prefix[wk.s] * H_kv + (long long)wk.g * wk.n;
    Walker wl;
    wl.start(u1 - 1, sm_prefix, NW, H_kv);
    const long long last_sb = (long long)sm_prefix[wl.s] * H_kv + (long long)wl.g * wl.n;
    sm_split[0] = make_split(wk.s, wk.g, first_sb, first_sb + wk.n);
    sm_split[1] = make_split(wl.s, wl.g, last_sb, last_sb + wl.n);
    sm_split_flags[0] = first_sb < u0 && first_sb != last_sb;  // split, and not also the last
    sm_split_flags[1] = last_sb < u0 || last_sb + wl.n > u1;
  }
  cp_async_wait_all();
  if constexpr (FP8) convert_own_q(0);
  __syncwarp();
  named_barrier(kConsumerBarrier, kConsumerThreads);
#pragma unroll
  for (int k = 1; k < kQSlots; ++k) {
    prefetch_or_skip(k, ahead);
    ahead = next_piece(ahead);
  }
  reset();
  set_limits(wk.s, wk.g);
  // Ring ownership: unit i of the range (i = u - u0) sits in slot i % stages,
  // and slot r belongs to consumer warp r % 4, so each warp waits on its
  // slots' phases strictly in order (a parity wait cannot tell phase k from
  // k - 2) whatever the ring depth.  A warp steps from one of its units
  // straight to its next: slot + 4 in the same round of the ring, else slot
  // `warp` of the next round.
  const int n_stages = p.stages;
  long long own_i = warp;  // this warp's next unit (index within the range)
  int own_slot = warp;
  uint32_t own_phase = 0;
  auto own_step = [&](long long& i, int& slot, uint32_t& ph) {
    if (slot + kConsumerWarps < n_stages) {
      i += kConsumerWarps;
      slot += kConsumerWarps;
    } else {
      i += n_stages - slot + warp;
      slot = warp;
      ph ^= 1u;
    }
  };
  const long long n_units = u1 - u0;
  long long ia = 0;  // the current piece's first unit (index within the range)
  for (;;) {
    const int s = wk.s, g = wk.g, n = wk.n, p0 = wk.p;
    const int sq = multi && QC > 1 ? s % N : s;  // the walked sequence's sequence
    const int len = sm_len[sq];  // read once per piece (the page waits below clobber memory)
    const long long ib = min(n_units, ia + (n - p0));  // one past its last unit here
    while (own_i < ib) {
      const int pg = p0 + (int)(own_i - ia);  // page of the sequence
      if constexpr (FP8) {
        if (!abort) {
          const bool ready = __all_sync(0xffffffffu, mbar_wait(&full_bar[own_slot], own_phase));
          if (!ready) {
            if (lane == 0) report(kStatusTimeout);
            abort = true;
          } else {
            const int valid = min(BS, len - pg * BS);
            uint8_t* st = smem + own_slot * kStageBytes;
            // Only the piece's last page can end early: zero its V rows past
            // the sequence (they may hold anything) so the V operand needs no mask.
            const bool tail = valid < BS;
            if (tail) {
              const int chunks = (BS - valid) * L::kHalves * 8;  // 16-byte chunks
              for (int c = lane; c < chunks; c += 32) {
                const int r = valid + c / (L::kHalves * 8);
                const int h = (c / 8) % L::kHalves;
                *reinterpret_cast<uint4*>(st + kPageBytes + h * kTileBytes + r * 128 +
                                          (c % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
              }
              __syncwarp();
            }
            // Fused cache append (FP8 caches): the piece's last page holds the new
            // token.  Its bf16 K and V rows (prefetched with the query group) are
            // quantized here as the standalone append does -- float f = max|x| /
            // 448 (1 for a zero row), byte = e4m3(x / f) rounded to nearest even,
            // saturating -- patched into the page and its row floats in shared
            // memory, and stored to the cache after the page is processed.
            // (head_dim 128 only: at 256 the code would cost the page loop a spill,
            // and the library runs the append as its own launch instead)
            const bool patch = kFp8FusedAppend && !multi && p.k_new != nullptr && pg == n - 1;
            constexpr int kE = D / 32;  // values of a row per lane
            const uint8_t* extra = sm_q + qbuf * kQSlotBytes + kAppendOff;  // k row, v row, block
            // byte lane * kE of row `slot`: 16-byte chunk c (128-byte half c / 8,
            // swizzled position c ^ slot % 8 within it), offset o in the chunk
            auto patch_off = [&](int slot) {
              const int c = (lane * kE) >> 4, o = (lane * kE) & 15;
              return (c >> 3) * kTileBytes + slot * 128 + (((c & 7) ^ (slot & 7)) << 4) + o;
            };
            if constexpr (kFp8FusedAppend) {
              if (patch) {
                fp8_patch_row<D>(extra, st, kPageBytes, kTileBytes, valid - 1,
                                 sm_scales + (size_t)own_slot * 2 * BS, BS, lane);
                __syncwarp();
              }
            }
            const uint32_t sc = smem_addr(sm_scales + (size_t)own_slot * 2 * BS);
            const uint32_t q16 = smem_addr(sm_q + qbuf * kQSlotBytes + kQTileBytes);
            const uint32_t k0 = smem_addr(st), v0 = smem_addr(st + kPageBytes);
            if constexpr (BS == 16) {
              const Tile8 t[1] = {{k0, v0, sc, sc + 4 * BS, valid}};
              process_fp8(std::integral_constant<int, 1>(), t, q16);
            } else {  // the two 16-token halves of a 32-token page
              const Tile8 t[2] = {{k0, v0, sc, sc + 4 * BS, min(16, valid)},
                                  {k0 + 16 * 128, v0 + 16 * 128, sc + 4 * 16, sc + 4 * (BS + 16),
                                   max(0, valid - 16)}};
              process_fp8(std::integral_constant<int, 2>(), t, q16);
            }
            // the zeroing's and the patch's generic writes precede the next tensor
            // copy into the slot
            if (tail || patch) fence_proxy_async_shared();
            if (kFp8FusedAppend && patch) {  // the patched bytes and floats, read back from the slot
              const int slot = valid - 1;
              const int new_block = *reinterpret_cast<const int*>(extra + 4 * D);
              if (p.num_blocks <= 0 || (new_block >= 0 && (long long)new_block < p.num_blocks)) {
                const size_t row = ((size_t)new_block * H_kv + g) * BS + slot;
                const int off = patch_off(slot);
                uint8_t* k8 = reinterpret_cast<uint8_t*>(p.k_cache) + row * D + lane * kE;
                uint8_t* v8 = reinterpret_cast<uint8_t*>(p.v_cache) + row * D + lane * kE;
                if constexpr (kE == 4) {
                  *reinterpret_cast<uint32_t*>(k8) = *reinterpret_cast<const uint32_t*>(st + off);
                  *reinterpret_cast<uint32_t*>(v8) =
                      *reinterpret_cast<const uint32_t*>(st + kPageBytes + off);
                } else {
                  *reinterpret_cast<uint2*>(k8) = *reinterpret_cast<const uint2*>(st + off);
                  *reinterpret_cast<uint2*>(v8) =
                      *reinterpret_cast<const uint2*>(st + kPageBytes + off);
                }
                if (lane == 0) {
                  const_cast<float*>(p.k_scale)[row] = sm_scales[(size_t)own_slot * 2 * BS + slot];
                  const_cast<float*>(p.v_scale)[row] =
                      sm_scales[(size_t)own_slot * 2 * BS + BS + slot];
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[own_slot]);
          }
        }
        own_step(own_i, own_slot, own_phase);
      } else {
        if (!abort) {
          // Fused cache append: the last page of a piece holds the sequence's
          // new token.  Its rows (prefetched with the piece's query group) are
          // patched into the page in shared memory once the page has landed
          // (the tensor copy brought whatever the cache held) and stored to the
          // cache for later calls.  This page is read by this CTA alone.
          const bool patch = !XP && !multi && p.k_new != nullptr && pg == n - 1;
          // Lanes poll the barrier independently; the vote both reconverges
          // the warp before the warp-collective ldmatrix / movmatrix / mma and
          // makes the outcome uniform.
          const bool ready = __all_sync(0xffffffffu, mbar_wait(&full_bar[own_slot], own_phase));
          if (!ready) {
            if (lane == 0) report(kStatusTimeout);
            abort = true;
          } else {
            const int valid = min(BS, len - pg * BS);
            uint8_t* st = smem + own_slot * kStageBytes;
            const uint8_t* extra = sm_q + qbuf * kQSlotBytes + kAppendOff;  // k row, v row, block
            if (patch) {
              const int slot = valid - 1;  // the new token, t = L - 1
              if (lane < D / 8) {
                // 16-byte chunk `lane` of the row: half lane / 8, swizzled position within it
                const int off =
                    (lane >> 3) * kTileBytes + slot * 128 + (((lane & 7) ^ (slot & 7)) << 4);
                *reinterpret_cast<uint4*>(st + off) = reinterpret_cast<const uint4*>(extra)[lane];
                *reinterpret_cast<uint4*>(st + kPageBytes + off) =
                    reinterpret_cast<const uint4*>(extra + 2 * D)[lane];
              }
              __syncwarp();
            }
            process_page(st, st + kPageBytes, sm_q + qbuf * kQSlotBytes, valid, pg * BS, lim);
            if (patch) {
              // the patch's generic writes precede the next tensor copy into this slot
              fence_proxy_async_shared();
              const int slot = valid - 1;
              const int new_block = *reinterpret_cast<const int*>(extra + 4 * D);
              if (lane < D / 8 &&
                  (p.num_blocks <= 0 || (new_block >= 0 && (long long)new_block < p.num_blocks))) {
                const size_t dst = (((size_t)new_block * H_kv + g) * BS + slot) * D + lane * 8;
                *reinterpret_cast<uint4*>(p.k_cache + dst) =
                    reinterpret_cast<const uint4*>(extra)[lane];
                *reinterpret_cast<uint4*>(p.v_cache + dst) =
                    reinterpret_cast<const uint4*>(extra + 2 * D)[lane];
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[own_slot]);
          }
        }
        own_step(own_i, own_slot, own_phase);
      }
    }
    const bool last = ib == n_units;
    if (!last) wk.advance((int)(ib - ia), sm_prefix, NW, H_kv);  // to the next piece
    ia = ib;
    const long long sb = (long long)sm_prefix[s] * H_kv + (long long)g * n;
    if (!last) {
      // A split piece that is not the range's last is its first: store its
      // partial, then arrive and publish at once with a release add (the
      // barrier below orders every thread's stores before it); the old value
      // is only read at the end of the range.
      const bool split = sb < u0;
      merge_warps(nullptr, nullptr);
      emit(s, g, split ? p.partials + (size_t)my_slot(sb) * R * kPartialRow : nullptr);
      // The next piece's query group is the oldest of the kQSlots - 1 groups in
      // flight: wait for it alone and make every thread's copies visible (FP8:
      // after converting its own to f16), then prefetch into the slot just
      // freed the piece kQSlots - 1 further on.
      const int qnext = qbuf + 1 == kQSlots ? 0 : qbuf + 1;
      cp_async_wait_group<kQSlots - 2>();
      if constexpr (FP8) convert_own_q(qnext);
      __syncwarp();
      named_barrier(kConsumerBarrier, kConsumerThreads);
      if (ctid == 0 && split)
        first_old = atom_add_release_gpu(p.counters + sm_split[0].c_first, 1 + (1 << 16));
      prefetch_or_skip(qbuf, ahead);
      ahead = next_piece(ahead);
      qbuf = qnext;
      reset();
      set_limits(wk.s, wk.g);
      continue;
    }
    // ---- the range's last piece.  When it is split, thread 0 arrives as soon
    // as the pages are done (before anything is stored); the last CTA to arrive
    // combines, keeping its own merged state in shared memory, while the
    // others store theirs and publish it.
    const Split xf = sm_split[0], xl = sm_split[1];
    const bool first_split = sm_split_flags[0] != 0, last_split = sm_split_flags[1] != 0;
    int* const word_f = p.counters + xf.c_first;  // [15:0] arrived, [31:16] published
    int* const word_l = p.counters + xl.c_first;
    const int n_f = xf.c_last - xf.c_first + 1;   // contributors
    const int n_l = xl.c_last - xl.c_first + 1;
    int old_l = 0;
    merge_warps(last_split ? word_l : nullptr, &old_l);
    if (!last_split) emit(s, g, nullptr);
    if (ctid == 0) {
      sm_flag[0] = first_split && (first_old & 0xffff) == n_f - 1 ? 1 : 0;
      sm_flag[1] = last_split && (old_l & 0xffff) == n_l - 1 ? 1 : 0;
    }
    __syncwarp();
    // A CTA whose page wait ran out (status bit 2; its state is garbage) still
    // stores, publishes and combines like the others, so every split's counter
    // completes and is reset: the workspace stays fit for the next call.
    named_barrier(kConsumerBarrier, kConsumerThreads);
    const bool cf = sm_flag[0] != 0, cl = sm_flag[1] != 0;
    // this CTA's part of the last piece: its place among the split's parts, and
    // whether the combine can take it from the ring instead of the workspace
    const int local_t = (int)blockIdx.x - xl.c_first;
    const int part_bytes = R * kPartialRow * 4;
    const bool local = cl && local_t < (p.stages * kStageBytes) / part_bytes;
    if (last_split && !local) {
      emit(s, g, p.partials + (size_t)my_slot(sb) * R * kPartialRow);
      __syncwarp();
      named_barrier(kConsumerBarrier, kConsumerThreads);
      if (ctid == 0) {
        if (!cl)
          atom_add_release_gpu(word_l, 1 << 16);  // publish
        else
          __threadfence();  // this CTA's stores, read back by its own bulk copies
      }
    }
    if (local) emit(s, g, reinterpret_cast<float*>(smem + local_t * part_bytes));
    if (!cf && !cl) break;
    if (ctid == 0) {
      bool ok = true;
#ifdef PAGED_ATTN_WAIT_TEST
      const int extra = p.test_skip_publish > 0 ? 1 : 0;  // one part more than exist
#else
      constexpr int extra = 0;
#endif
      if (cl) ok = wait_published(word_l, n_l - 1 + extra);  // every other part
      if (cf && ok) ok = wait_published(word_f, n_f + extra);
      if (!ok) report(kStatusTimeout);
      sm_flag[2] = ok ? 1 : 0;
    }
    __syncwarp();
    named_barrier(kConsumerBarrier, kConsumerThreads);  // also orders the ring writes
    if (sm_flag[2] == 0) break;
    if (cl)
      combine(xl, xf, cf ? 2 : 1, local ? local_t : -1);
    else
      combine(xf, xf, 1, -1);
    if (ctid == 0) {  // ready for the next call
      if (cf) *word_f = 0;
      if (cl) *word_l = 0;
    }
    break;
  }
  cp_async_wait_all();
}

}  // namespace pagedattn
