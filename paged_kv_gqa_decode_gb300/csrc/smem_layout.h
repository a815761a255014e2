// Shared-memory layout of the decode kernel, as plain C++ so the host plan, the
// kernel and a host-only alignment check all use the same arithmetic.
//
// The pipeline ring starts the (1024-byte aligned) dynamic shared memory, as the
// 128-byte TMA swizzle requires; every later region starts on a 128-byte
// boundary, so mbarriers (8 bytes), ldmatrix rows and cp.async chunks (16) and
// the float4 merge buffer (16) are aligned whatever the ring depth, the group
// size or the batch.
#pragma once

#if defined(__CUDACC__)
#define PAGEDATTN_HD __host__ __device__
#else
#define PAGEDATTN_HD
#endif

namespace pagedattn {

constexpr int kConsumerWarps = 4;
// Query slots: the current piece's query group and the next kQSlots - 1 pieces'
// (prefetched ahead, so a run of short pieces does not wait on each fetch).
constexpr int kQSlots = 2;

PAGEDATTN_HD constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// FP8: the caches hold e4m3 bytes (head_dim 128 or 256) plus one float per
// cache row for K and for V.
template <int D, int BS, bool FP8 = false>
struct SmemLayout {
  static constexpr int kElem = FP8 ? 1 : 2;           // bytes per cache element
  static constexpr int kHalves = D * kElem / 128;     // 128-byte column halves of a row
  static constexpr int kTileBytes = BS * 128;         // one half of one page
  static constexpr int kPageBytes = kHalves * kTileBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;  // K page + V page
  static constexpr int kScaleBytes = FP8 ? 2 * BS * 4 : 0;  // a stage's K and V row floats
  static constexpr int kRowStride = D + 4;            // padded fp32 row in the merge buffer
  static constexpr int kQ16Stride = 2 * D + 32;       // FP8: padded f16 query row

  int stages, G, num_seqs;  // G: query rows of one piece (the group size, or a chunk)
  int qo_entries = 0;       // multi-token decode: num_seqs + 1 query-row offsets
  int walks = 1;            // multi-token decode: passes over the sequences (row chunks)
  // [0, bars): the ring of `stages` K/V pages (at the end of a range it holds the
  // partial states being combined); then the mbarriers full[stages],
  // empty[stages] and one for the combine's copies; FP8: the ring of row floats
  PAGEDATTN_HD int bars() const { return stages * kStageBytes; }
  PAGEDATTN_HD int scales() const { return align_up(bars() + (2 * stages + 1) * 8, 128); }
  PAGEDATTN_HD int merge_m() const { return align_up(scales() + stages * kScaleBytes, 128); }
  PAGEDATTN_HD int merge_l() const { return merge_m() + kConsumerWarps * 16 * 4; }
  PAGEDATTN_HD int final_ml() const { return merge_l() + kConsumerWarps * 16 * 4; }
  PAGEDATTN_HD int flag() const { return final_ml() + 32 * 4; }  // a few ints
  PAGEDATTN_HD int merge_o() const { return flag() + 128; }
  // one query tile: the group's rows padded to 8 (G <= 8) or 16 heads
  PAGEDATTN_HD int q_rows() const { return G > 8 ? 16 : 8; }
  PAGEDATTN_HD int q_tile_bytes() const { return q_rows() * D * 2; }
  // one query slot: the bf16 tile, then (FP8) the tile as f16, then (fused cache
  // append) the piece's new K row, new V row (bf16) and the block id of its last
  // page
  PAGEDATTN_HD int q_f16_bytes() const { return FP8 ? q_rows() * kQ16Stride : 0; }
  PAGEDATTN_HD int q_extra_bytes() const { return q_f16_bytes() + 4 * D + 16; }
  PAGEDATTN_HD int q_slot_bytes() const {
    return align_up(q_tile_bytes() + q_extra_bytes(), 128);
  }
  PAGEDATTN_HD int qtile() const {  // kQSlots query slots
    return merge_o() + align_up(kConsumerWarps * G * kRowStride * 4, 128);
  }
  PAGEDATTN_HD int prefix() const { return qtile() + kQSlots * q_slot_bytes(); }
  // the page prefix of each pass, then the same prefix with each (sequence, KV
  // head) piece weighted by its fixed cost (the work split's positions)
  PAGEDATTN_HD int wprefix() const { return prefix() + align_up((walks * num_seqs + 1) * 4, 128); }
  PAGEDATTN_HD int lens() const { return wprefix() + align_up((walks * num_seqs + 1) * 4, 128); }
  PAGEDATTN_HD int qo() const { return align_up(lens() + num_seqs * 4, 16); }
  PAGEDATTN_HD int total() const { return qo() + qo_entries * 4; }
};

}  // namespace pagedattn
