// Split-KV paged GQA decode attention for GB300 (sm_103a).
//
// What it computes is the operation of include/paged_attn.h ("Paged Attention
// Kernel Architecture for BI-V100", section 1; paging layout and head map of
// the RL.cu "Add Cuda Kernel" tutorial's paged decode).  How:
//
//  * Work split (section 6 of the BI-V100 design splits each sequence into
//    fixed 512-token partitions; here the split is re-derived for ragged
//    batches): the units of work are pages (s, g, p) -- one physical block of
//    one KV head.  Flattened in (s, g, p) order they are cut into C equal
//    contiguous ranges, one per persistent CTA (C = number of SMs, reduced so
//    each CTA gets at least kMinPagesPerCta pages).  Every CTA streams the same
//    number of bytes whatever the length mix, and a range crossing (s, g)
//    boundaries simply produces one partial softmax state per piece.
//
//  * Data movement: one producer warp walks the range, reads the block table
//    and issues TMA tiled loads (cp.async.bulk.tensor.3d) of each K and V page
//    into a ring of shared-memory stages, 128-byte swizzled, completing on an
//    mbarrier per stage.  Each page of one KV head is one contiguous
//    block_size x head_dim run in HBM; the 3-D tensor map addresses it as
//    (column, g * block_size, physical block).
//
//  * Math: consumer warps take pages round-robin.  The whole GQA group of the
//    KV head (G <= 16 query heads, zero-padded to 16 rows) is the A operand of
//    bf16 m16n8k16 tensor-core MMAs: S = Q K^T over the page (K read with
//    ldmatrix from the swizzled tile), online softmax in fp32 on the
//    accumulator fragments (BI-V100 design, section 2, Level 1: running max,
//    exp-sum and weighted V), then O += P V (V read with ldmatrix.trans).  So
//    every K/V byte leaves HBM once and feeds all G heads.
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

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace pagedattn {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kMinPagesPerCta = 8;
constexpr int kMaxStages = 16;
constexpr int kConsumerBarrier = 1;

// Status bits written to the workspace / caller status word.
constexpr int kStatusBadBlock = 1;
constexpr int kStatusBadLength = 2;
constexpr int kStatusTimeout = 4;

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
};

// Shared-memory layout, in bytes from a 1024-aligned base.
template <int D, int BS>
struct SmemLayout {
  static constexpr int kHalves = D / 64;              // 128-byte column halves of a row
  static constexpr int kTileBytes = BS * 128;         // one half of one page
  static constexpr int kPageBytes = kHalves * kTileBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;  // K page + V page
  static constexpr int kRowStride = D + 8;            // padded fp32 row in the merge buffer

  int stages, G, num_seqs;
  __host__ __device__ int bars() const { return stages * kStageBytes; }
  __host__ __device__ int merge_m() const { return bars() + 2 * stages * 8; }
  __host__ __device__ int merge_l() const { return merge_m() + kConsumerWarps * 16 * 4; }
  __host__ __device__ int final_ml() const { return merge_l() + kConsumerWarps * 16 * 4; }
  __host__ __device__ int flag() const { return final_ml() + 32 * 4; }
  __host__ __device__ int merge_o() const { return flag() + 16; }
  __host__ __device__ int prefix() const {
    return merge_o() + kConsumerWarps * G * kRowStride * 4;
  }
  __host__ __device__ int lens() const { return prefix() + (num_seqs + 1) * 4; }
  __host__ __device__ int total() const { return lens() + num_seqs * 4; }
};

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
    g = (int)(off / n);
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
};

// The CTA whose range contains unit u, for ranges [floor(c W / C), floor((c+1) W / C)).
__device__ __forceinline__ int cta_of(long long u, long long W, long long C) {
  return (int)(((u + 1) * C - 1) / W);
}

__device__ __forceinline__ long long range_begin(long long c, long long W, long long C) {
  return c * W / C;
}

template <int D, int BS, bool G16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using L = SmemLayout<D, BS>;
  constexpr int kTileBytes = L::kTileBytes;
  constexpr int kPageBytes = L::kPageBytes;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int kRowStride = L::kRowStride;
  constexpr int kPartialRow = D + 4;  // [M, L, pad, pad, o[0..D)]
  constexpr int kNT = D / 8;          // n8 tiles across head_dim
  constexpr int kKT = D / 16;         // k16 steps across head_dim
  constexpr int kST = BS / 8;         // n8 token tiles per page

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const L lay{p.stages, p.G, p.num_seqs};
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + lay.bars());
  uint64_t* empty_bar = full_bar + p.stages;
  float* sm_m = reinterpret_cast<float*>(smem + lay.merge_m());
  float* sm_l = reinterpret_cast<float*>(smem + lay.merge_l());
  float* sm_final = reinterpret_cast<float*>(smem + lay.final_ml());  // [0,16) M, [16,32) L
  int* sm_flag = reinterpret_cast<int*>(smem + lay.flag());
  float* sm_o = reinterpret_cast<float*>(smem + lay.merge_o());
  int* sm_prefix = reinterpret_cast<int*>(smem + lay.prefix());
  int* sm_len = reinterpret_cast<int*>(smem + lay.lens());

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int N = p.num_seqs;
  const int H_kv = p.H_kv;
  const int G = p.G;
  const int cap = p.maxb * BS;

  // ---- 1. clamped lengths and the exclusive prefix of pages per sequence
  {
    const int per = (N + kThreads - 1) / kThreads;
    const int s0 = tid * per;
    const int s1 = min(N, s0 + per);
    int local = 0;
    for (int s = s0; s < s1; ++s) {
      int len = __ldg(p.seq_lens + s);
      if (len < 0 || len > cap) {
        if (p.num_blocks > 0 && blockIdx.x == 0) atomicOr(p.status, kStatusBadLength);
        len = min(max(len, 0), cap);
      }
      sm_len[s] = len;
      local += (len + BS - 1) / BS;
    }
    // block-wide exclusive scan of `local`
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_tot[kThreads / 32];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int s = s0; s < s1; ++s) {
      sm_prefix[s] = run;
      run += (sm_len[s] + BS - 1) / BS;
    }
    if (tid == kThreads - 1) sm_prefix[N] = base + incl;
    __syncthreads();
  }

  // ---- 2. empty sequences get zero rows (spread over CTAs)
  for (int s = blockIdx.x; s < N; s += gridDim.x) {
    if (sm_len[s] != 0) continue;
    uint32_t* o32 = reinterpret_cast<uint32_t*>(p.out + (size_t)s * p.H_q * D);
    for (int i = tid; i < p.H_q * D / 2; i += kThreads) o32[i] = 0u;
  }

  const long long W = (long long)sm_prefix[N] * H_kv;
  if (W == 0) return;
  const long long C =
      min((long long)gridDim.x, max(1LL, (W + kMinPagesPerCta - 1) / kMinPagesPerCta));
  if ((long long)blockIdx.x >= C) return;
  const long long u0 = range_begin(blockIdx.x, W, C);
  const long long u1 = range_begin(blockIdx.x + 1, W, C);
  if (u0 >= u1) return;

  if (tid == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // =================================================================== producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const uint64_t policy = l2_evict_first_policy();
    Walker wk;
    if (u0 + lane < u1) wk.start(u0 + lane, sm_prefix, N, H_kv);
    auto fetch = [&](long long u) -> int2 {
      // physical block and KV head of this lane's unit (block -1 past the range)
      if (u >= u1) return make_int2(-1, 0);
      int pb = __ldg(p.block_tables + (size_t)wk.s * p.maxb + wk.p);
      if (p.num_blocks > 0 && (pb < 0 || (long long)pb >= p.num_blocks))
        atomicOr(p.status, kStatusBadBlock);  // the TMA bounds check reads it as zeros
      return make_int2(pb, wk.g);
    };
    int2 cur = fetch(u0 + lane);
    int stage = 0;
    uint32_t phase = 0;
    bool abort = false;
    long long issued = 0;
    for (long long ub = u0; ub < u1 && !abort; ub += 32) {
      // advance this lane's walker to its unit of the next batch and start that load
      int2 nxt = make_int2(-1, 0);
      if (ub + 32 + lane < u1) {
        for (int k = 0; k < 32; ++k) wk.next(sm_prefix, N, H_kv);
        nxt = fetch(ub + 32 + lane);
      }
      const int cnt = (int)min(32LL, u1 - ub);
      for (int j = 0; j < cnt; ++j) {
        const int pb = __shfl_sync(0xffffffffu, cur.x, j);
        const int g = __shfl_sync(0xffffffffu, cur.y, j);
        if (lane == 0 && !abort) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u)) {
            atomicOr(p.status, kStatusTimeout);
            abort = true;
          } else {
            mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
            uint8_t* st = smem + stage * kStageBytes;
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
              tma_load_3d(st + hh * kTileBytes, &tm_k, &full_bar[stage], hh * 64, g * BS, pb,
                          policy);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
              tma_load_3d(st + kPageBytes + hh * kTileBytes, &tm_v, &full_bar[stage], hh * 64,
                          g * BS, pb, policy);
            ++issued;
          }
        }
        abort = __shfl_sync(0xffffffffu, abort, 0);
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      cur = nxt;
    }
    // Drain: make sure no tensor copy issued by this CTA is still in flight when it exits.
    if (lane == 0 && issued > 0) {
      const long long first = issued > p.stages ? issued - p.stages : 0;
      for (long long i = first; i < issued; ++i) {
        const int st = (int)(i % p.stages);
        const uint32_t ph = (uint32_t)((i / p.stages) & 1);
        if (!mbar_wait(&full_bar[st], ph)) {
          atomicOr(p.status, kStatusTimeout);
          break;
        }
      }
    }
    return;
  }

  // ===================================================================== consumers
  const int r0 = lane >> 2;       // accumulator row (query head within the group)
  const int cq = 2 * (lane & 3);  // column pair within an n8 tile
  const int ctid = tid;           // 0 .. kConsumerThreads-1

  uint32_t qa[kKT][G16 ? 4 : 2];  // A fragments of the query group
  float o_acc[kNT][G16 ? 4 : 2];  // output accumulator fragments
  float m_run[2], l_run[2];       // per accumulator row: running max (log2 domain) and sum

  auto load_q = [&](int s, int g) {
    const __nv_bfloat16* qb = p.q + ((size_t)s * p.H_q + (size_t)g * G) * D;
#pragma unroll
    for (int kk = 0; kk < kKT; ++kk) {
      const int c = kk * 16 + cq;
      const uint32_t* r0p = reinterpret_cast<const uint32_t*>(qb + (size_t)r0 * D + c);
      qa[kk][0] = r0 < G ? __ldg(r0p) : 0u;
      qa[kk][1] = r0 < G ? __ldg(r0p + 4) : 0u;
      if constexpr (G16) {
        const uint32_t* r1p = reinterpret_cast<const uint32_t*>(qb + (size_t)(r0 + 8) * D + c);
        qa[kk][2] = r0 + 8 < G ? __ldg(r1p) : 0u;
        qa[kk][3] = r0 + 8 < G ? __ldg(r1p + 4) : 0u;
      }
    }
  };
  auto reset = [&]() {
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < (G16 ? 4 : 2); ++e) o_acc[nt][e] = 0.f;
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
  };

  // One page: S = Q K^T, online softmax, O += P V.
  auto process_page = [&](const uint8_t* kt, const uint8_t* vt, int valid) {
    const uint32_t kbase = smem_addr(kt);
    const uint32_t vbase = smem_addr(vt);
    float s_acc[kST][4];
#pragma unroll
    for (int j = 0; j < kST; ++j) s_acc[j][0] = s_acc[j][1] = s_acc[j][2] = s_acc[j][3] = 0.f;

    // ---- S = Q K^T: B operand rows are tokens, 16-byte chunks of head_dim, swizzled
#pragma unroll
    for (int kq = 0; kq < D / 32; ++kq) {
      const int chunk = 4 * kq + (lane >> 3);
      const uint32_t koff = (uint32_t)((chunk >> 3) * kTileBytes +
                                       ((((chunk & 7) ^ (lane & 7))) << 4));
#pragma unroll
      for (int j = 0; j < kST; ++j) {
        const uint32_t addr = kbase + koff + (uint32_t)((8 * j + (lane & 7)) * 128);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        if constexpr (G16) {
          mma_bf16_16816(s_acc[j], qa[2 * kq][0], qa[2 * kq][2], qa[2 * kq][1], qa[2 * kq][3],
                         b0, b1);
          mma_bf16_16816(s_acc[j], qa[2 * kq + 1][0], qa[2 * kq + 1][2], qa[2 * kq + 1][1],
                         qa[2 * kq + 1][3], b2, b3);
        } else {
          mma_bf16_16816_top(s_acc[j][0], s_acc[j][1], qa[2 * kq][0], qa[2 * kq][1], b0, b1);
          mma_bf16_16816_top(s_acc[j][0], s_acc[j][1], qa[2 * kq + 1][0], qa[2 * kq + 1][1], b2,
                             b3);
        }
      }
    }

    // ---- online softmax (log2 domain); masked tokens are selected out
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < kST; ++j)
#pragma unroll
      for (int e = 0; e < (G16 ? 4 : 2); ++e) {
        const int tok = 8 * j + cq + (e & 1);
        const float x = tok < valid ? s_acc[j][e] * p.scale_log2 : -INFINITY;
        s_acc[j][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < (G16 ? 2 : 1); ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float m_new = fmaxf(m_run[h], mx[h]);
      alpha[h] = fast_exp2(m_run[h] - m_new);
      m_run[h] = m_new;
    }
    uint32_t pk[kST][2];  // P as packed bf16 pairs: [tile][row half]
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kST; ++j)
#pragma unroll
      for (int h = 0; h < (G16 ? 2 : 1); ++h) {
        const float e0 = fast_exp2(s_acc[j][2 * h] - m_run[h]);
        const float e1 = fast_exp2(s_acc[j][2 * h + 1] - m_run[h]);
        const uint32_t pr = pack_bf16x2(e0, e1);
        pk[j][h] = pr;
        psum[h] += bf16lo_to_f32(pr) + bf16hi_to_f32(pr);
      }
#pragma unroll
    for (int h = 0; h < (G16 ? 2 : 1); ++h) l_run[h] = l_run[h] * alpha[h] + psum[h];
    const bool rescale = G16 ? __any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)
                             : __any_sync(0xffffffffu, alpha[0] != 1.f);
    if (rescale) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        o_acc[nt][0] *= alpha[0];
        o_acc[nt][1] *= alpha[0];
        if constexpr (G16) {
          o_acc[nt][2] *= alpha[1];
          o_acc[nt][3] *= alpha[1];
        }
      }
    }

    // ---- O += P V: B operand from V rows (tokens) with a transposing ldmatrix
    const bool tail = valid < BS;
#pragma unroll
    for (int jj = 0; jj < BS / 16; ++jj) {
      const uint32_t a0 = pk[2 * jj][0];
      const uint32_t a2 = pk[2 * jj + 1][0];
      const uint32_t a1 = G16 ? pk[2 * jj][1] : 0u;
      const uint32_t a3 = G16 ? pk[2 * jj + 1][1] : 0u;
      uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
      if (tail) {  // rows past the sequence may hold anything: zero them in the fragment
        const int t0 = 16 * jj + cq;
        vmask_lo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
        vmask_hi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
      }
      const int i = lane >> 3;
      const int trow = 16 * jj + (lane & 7) + ((i & 1) << 3);
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        const int chunk = 2 * n2 + (i >> 1);
        const uint32_t addr = vbase + (uint32_t)((chunk >> 3) * kTileBytes + trow * 128 +
                                                 (((chunk & 7) ^ (lane & 7)) << 4));
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        b0 &= vmask_lo;
        b1 &= vmask_hi;
        b2 &= vmask_lo;
        b3 &= vmask_hi;
        if constexpr (G16) {
          mma_bf16_16816(o_acc[2 * n2], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o_acc[2 * n2 + 1], a0, a1, a2, a3, b2, b3);
        } else {
          mma_bf16_16816_top(o_acc[2 * n2][0], o_acc[2 * n2][1], a0, a2, b0, b1);
          mma_bf16_16816_top(o_acc[2 * n2 + 1][0], o_acc[2 * n2 + 1][1], a0, a2, b2, b3);
        }
      }
    }
  };

  // Merge the consumer warps' states for (s, g) and emit the output row block
  // (whole piece) or a partial state (split piece; the last piece combines).
  auto finish_piece = [&](int s, int g, long long sb, long long se) {
    const bool split = sb < u0 || se > u1;
#pragma unroll
    for (int h = 0; h < (G16 ? 2 : 1); ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    if ((lane & 3) == 0) {
      sm_m[warp * 16 + r0] = m_run[0];
      sm_l[warp * 16 + r0] = l_run[0];
      if constexpr (G16) {
        sm_m[warp * 16 + r0 + 8] = m_run[1];
        sm_l[warp * 16 + r0 + 8] = l_run[1];
      }
    }
    named_barrier(kConsumerBarrier, kConsumerThreads);
#pragma unroll
    for (int h = 0; h < (G16 ? 2 : 1); ++h) {
      const int r = r0 + 8 * h;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * 16 + r]);
      float Lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = sm_m[w * 16 + r];
        if (mw != -INFINITY) Lsum += sm_l[w * 16 + r] * fast_exp2(mw - M);
      }
      const float f = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - M);
      if (r < G) {
        float* row = sm_o + (warp * G + r) * kRowStride + cq;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          *reinterpret_cast<float2*>(row + 8 * nt) =
              make_float2(o_acc[nt][2 * h] * f, o_acc[nt][2 * h + 1] * f);
      }
      if (warp == 0 && (lane & 3) == 0) {
        sm_final[r] = M;
        sm_final[16 + r] = Lsum;
      }
    }
    named_barrier(kConsumerBarrier, kConsumerThreads);

    const long long C_ = C;
    float* mine = nullptr;
    if (split) {
      const int slot = 2 * blockIdx.x + (sb <= u0 ? 0 : 1);
      mine = p.partials + (size_t)slot * G * kPartialRow;
    }
    for (int i = ctid; i < G * (D / 2); i += kConsumerThreads) {
      const int r = i / (D / 2);
      const int d = 2 * (i - r * (D / 2));
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float2 v = *reinterpret_cast<const float2*>(sm_o + (w * G + r) * kRowStride + d);
        acc.x += v.x;
        acc.y += v.y;
      }
      if (!split) {
        const float inv = 1.f / sm_final[16 + r];
        *reinterpret_cast<uint32_t*>(p.out + ((size_t)s * p.H_q + (size_t)g * G + r) * D + d) =
            pack_bf16x2(acc.x * inv, acc.y * inv);
      } else {
        float* row = mine + r * kPartialRow;
        *reinterpret_cast<float2*>(row + 4 + d) = acc;
        if (d == 0) *reinterpret_cast<float2*>(row) = make_float2(sm_final[r], sm_final[16 + r]);
      }
    }
    if (split) {
      __threadfence();
      named_barrier(kConsumerBarrier, kConsumerThreads);
      const int c_first = cta_of(sb, W, C_);
      const int c_last = cta_of(se - 1, W, C_);
      if (ctid == 0) {
        // A split (s, g) is identified by the first CTA holding a piece of it: only
        // that CTA's last piece can run past its range, so the index is unique.
        const int old = atomicAdd(p.counters + c_first, 1);
        *sm_flag = (old == c_last - c_first) ? 1 : 0;
      }
      named_barrier(kConsumerBarrier, kConsumerThreads);
      if (*sm_flag) {
        __threadfence();
        for (int i = ctid; i < G * (D / 2); i += kConsumerThreads) {
          const int r = i / (D / 2);
          const int d = 2 * (i - r * (D / 2));
          float M = -INFINITY;
          for (int c = c_first; c <= c_last; ++c) {
            const int slot = 2 * c + (sb <= range_begin(c, W, C_) ? 0 : 1);
            M = fmaxf(M, __ldcg(p.partials + ((size_t)slot * G + r) * kPartialRow));
          }
          float den = 0.f, nx = 0.f, ny = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int slot = 2 * c + (sb <= range_begin(c, W, C_) ? 0 : 1);
            const float* row = p.partials + ((size_t)slot * G + r) * kPartialRow;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(row));
            const float2 o = __ldcg(reinterpret_cast<const float2*>(row + 4 + d));
            const float wgt = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
            den += wgt * ml.y;
            nx += wgt * o.x;
            ny += wgt * o.y;
          }
          const float inv = 1.f / den;
          *reinterpret_cast<uint32_t*>(p.out + ((size_t)s * p.H_q + (size_t)g * G + r) * D +
                                       d) = pack_bf16x2(nx * inv, ny * inv);
        }
        if (ctid == 0) p.counters[c_first] = 0;  // ready for the next call
      }
    }
    named_barrier(kConsumerBarrier, kConsumerThreads);
  };

  Walker wk;
  wk.start(u0, sm_prefix, N, H_kv);
  load_q(wk.s, wk.g);
  reset();
  int stage = 0;
  uint32_t phase = 0;
  int owner = 0;  // which consumer warp takes the current unit
  bool abort = false;
  for (long long u = u0; u < u1; ++u) {
    if (owner == warp && !abort) {
      if (!mbar_wait(&full_bar[stage], phase)) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        abort = true;
      } else {
        const int valid = min(BS, sm_len[wk.s] - wk.p * BS);
        const uint8_t* st = smem + stage * kStageBytes;
        process_page(st, st + kPageBytes, valid);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
      }
    }
    if (++owner == kConsumerWarps) owner = 0;
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }
    const int s = wk.s, g = wk.g, n = wk.n;
    const bool last = u + 1 == u1;
    wk.next(sm_prefix, N, H_kv);
    if (last || wk.g != g || wk.s != s) {
      const long long sb = (long long)sm_prefix[s] * H_kv + (long long)g * n;
      finish_piece(s, g, sb, sb + n);
      if (!last) {
        load_q(wk.s, wk.g);
        reset();
      }
    }
  }
}

}  // namespace pagedattn
