/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-KV GQA decode attention library.
 *
 * The operation (every entry point below computes it):
 *
 *   "Paged Attention Kernel Architecture for BI-V100", section 1 (Problem
 *   Definition): for one new query token per sequence,
 *       out[s, h, :] = softmax_t( scale * q[s, h, :] . K_t ) . V_t,   t < seq_lens[s],
 *   where K_t / V_t are rows of a paged cache reached through a block table.
 *   Layout, length meaning and GQA head map follow the "Add Cuda Kernel"
 *   tutorial (RL.cu), include/kernels/attention.cuh, "Paged Attention - Decode":
 *       K_t = k_cache[block_tables[s, t / block_size], g, t % block_size, :]
 *       g   = h * H_kv / H_q          (H_q must be a multiple of H_kv; G = H_q / H_kv)
 *   The caller passes `scale` (the tutorial's launcher recomputed 1/sqrt(head_dim)
 *   and ignored its argument; here the argument is used as given).
 *
 * Tensors (DEVICE-ADDRESSABLE pointers, owned by the caller, densely packed
 * row-major, base addresses 16-byte aligned).  The caches (and their row floats)
 * must be device memory.  Every other tensor -- q, out, block_tables, seq_lens,
 * qo_indptr, the new K/V rows of the appends, status words -- may also be
 * pinned host memory (cudaMallocHost / cudaHostAlloc, which unified addressing
 * makes directly addressable from the device): the kernels then read and write
 * it over the host link (NVLink-C2C on GB300) inside the call, with no separate
 * copy, and the results are the same bits.  The library never dereferences any
 * of these pointers on the host.
 *   q            [num_seqs, H_q, head_dim]                      bf16   (read)
 *   k_cache      [num_blocks, H_kv, block_size, head_dim]       bf16   (read)
 *   v_cache      [num_blocks, H_kv, block_size, head_dim]       bf16   (read)
 *   out          [num_seqs, H_q, head_dim]                      bf16   (written)
 *   block_tables [num_seqs, max_blocks_per_seq]                 int32  (read)
 *   seq_lens     [num_seqs]                                     int32  (read)
 *
 * seq_lens[s] is the number of cached tokens the query attends to (the new
 * token's K/V must already be in the cache).  A length of 0 writes a zero row.
 * Lengths are clamped to [0, max_blocks_per_seq * block_size].  Only the
 * first ceil(seq_lens[s] / block_size) entries of a block-table row are read,
 * and only the rows t < seq_lens[s] of those blocks: slots past the end may
 * hold anything, NaN included.
 *
 * Supported: head_dim in {64, 128, 256}; block_size in {16, 32}; 1 <= G <= 16;
 * num_seqs >= 0 (0 is a no-op).  Arithmetic: bf16 inputs, fp32 accumulation
 * (tensor-core products of bf16 operands), bf16 output rounded to nearest even.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream), never synchronises, and never allocates except
 * where an entry point says so.  Block ids outside the caller's pool are not
 * detected unless checks are on: paged_attn_decode_checked checks its own
 * call, and paged_attn_set_checks turns the same checks on for every later
 * call of the calling thread (all decode and append entry points).
 *
 * Errors: every entry point returns PAGED_ATTN_OK (0) or a negative
 * PAGED_ATTN_ERR_* code.  Argument errors are detected on the host before any
 * CUDA call.  Nothing aborts, throws or exits.
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Only the entry points below are exported from the shared library (it is built
 * with hidden default visibility), so several copies of it -- say, two versions
 * -- can live in one process without sharing any internal state. */
#if defined(__GNUC__)
#define PAGED_ATTN_API __attribute__((visibility("default")))
#else
#define PAGED_ATTN_API
#endif

#define PAGED_ATTN_OK 0
#define PAGED_ATTN_ERR_POINTER (-1)    /* null or not 16-byte aligned pointer */
#define PAGED_ATTN_ERR_HEADS (-2)      /* H_kv <= 0, H_q % H_kv != 0, or G > 16 */
#define PAGED_ATTN_ERR_HEAD_DIM (-3)   /* head_dim not in {64, 128, 256} */
#define PAGED_ATTN_ERR_BLOCK_SIZE (-4) /* block_size not in {16, 32} */
#define PAGED_ATTN_ERR_SIZES (-5)      /* num_seqs < 0, max_blocks_per_seq <= 0, or too large */
#define PAGED_ATTN_ERR_CUDA (-6)       /* a CUDA runtime/driver call failed; see paged_attn_last_cuda_error */
#define PAGED_ATTN_ERR_WORKSPACE (-7)  /* workspace pointer null/misaligned or smaller than required */
#define PAGED_ATTN_ERR_SCALE (-8)      /* scale is not finite */
#define PAGED_ATTN_ERR_STATIC_SCRATCH (-9) /* sizes exceed paged_attn_decode_static's scratch */
#define PAGED_ATTN_ERR_FLAGS (-10)     /* unknown bits in paged_attn_set_launch_flags */

/* Launch flags (paged_attn_set_launch_flags). */
#define PAGED_ATTN_FLAG_EARLY_PROLOGUE 1

/*
 * Decode attention (the operation above).
 *
 * Scratch: the split-KV partial states live in a per-device workspace that the
 * library owns.  The first call on a device (and any call that needs a larger
 * workspace than before) allocates it with cudaMallocAsync on `stream` from the
 * device's default memory pool and zero-fills it there (a smaller one is
 * released with cudaFreeAsync on `stream`, after the calls before it on that
 * stream); later calls allocate nothing.  Because the workspace is shared,
 * calls that may overlap on the GPU (different streams, same device) race:
 * give each concurrent stream its own workspace through paged_attn_decode_ws.
 */
PAGED_ATTN_API int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int H_q, int H_kv, int head_dim, int max_blocks_per_seq, int block_size,
                      float scale, void* stream);

/*
 * Bytes of caller-provided workspace that paged_attn_decode_ws needs for these
 * sizes on the CURRENT device (it depends on the device's SM count).  Returns 0
 * for unsupported sizes.
 */
PAGED_ATTN_API size_t paged_attn_workspace_bytes(int num_seqs, int H_q, int H_kv, int head_dim,
                                  int max_blocks_per_seq, int block_size);

/*
 * Same operation with a caller-owned device workspace of at least
 * paged_attn_workspace_bytes(...) bytes, 256-byte aligned.  The workspace
 * must be zero-filled before its first use; every call that returns
 * PAGED_ATTN_OK and completes on the GPU leaves its counter region (whose
 * place depends only on the device) zero again, so the same workspace serves
 * any later call on the same device that fits in it.  Calls sharing one
 * workspace must not overlap on the GPU.  Allocates nothing.
 */
PAGED_ATTN_API int paged_attn_decode_ws(const void* q, const void* k_cache, const void* v_cache, void* out,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                         int H_q, int H_kv, int head_dim, int max_blocks_per_seq, int block_size,
                         float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Same operation with device-side input checks.  num_blocks is the size of the
 * caller's block pool.  A block id outside [0, num_blocks) in a used table
 * entry, or a sequence length outside [0, max_blocks_per_seq * block_size],
 * sets bit 0 (bad block) or bit 1 (bad length) of *d_status (a device int32
 * the caller zero-fills); bad blocks read as zero rows, bad lengths are
 * clamped, and no memory outside the pool is read.  Bit 2 reports that a
 * pipeline wait in the kernel ran out of its iteration limit and bit 3 that
 * the kernel rejected its launch configuration (library faults, never
 * expected; the output of such a call is undefined, the workspace stays
 * usable unless a combine wait ran out, in which case the workspace must be
 * zero-filled again before its next use: paged_attn_reset_workspace for the
 * library-owned one).  The
 * kernel writes *d_status only after the work ahead of it in the stream has
 * completed, so that work may zero-fill it.  Uses the library-owned workspace
 * like paged_attn_decode.
 */
PAGED_ATTN_API int paged_attn_decode_checked(const void* q, const void* k_cache, const void* v_cache, void* out,
                              const int32_t* block_tables, const int32_t* seq_lens,
                              int num_seqs, int H_q, int H_kv, int head_dim,
                              int max_blocks_per_seq, int block_size, float scale,
                              long long num_blocks, int32_t* d_status, void* stream);

/*
 * Same operation for callers that cannot allocate device memory.  There is no
 * counterpart in the reference pages; this entry point exists for callers whose
 * host framework owns all device memory -- a serving engine that reserves the
 * whole HBM for its KV-cache pool, or a plugin host that forbids allocation --
 * and for decode loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  It calls no cudaMalloc, cudaFree or allocating library
 * routine: its scratch (split-KV partial states and combine counters) is a
 * fixed 4 MiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits.  Sizes whose scratch would exceed
 * 4 MiB (those for which paged_attn_workspace_bytes() reports more) return
 * PAGED_ATTN_ERR_STATIC_SCRATCH before anything is launched (on a 152-SM
 * GB300 that is, for instance, head_dim 128 with 16 query heads per KV head;
 * the LLaMA-3-8B-, Qwen- and GQA-8-shaped decode batches all fit).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it, so make that first call before any
 * stream capture.  Every call clears the array's status and counter region
 * on `stream` (a memset, not an allocation) and then shares the array: calls
 * that may overlap on the GPU (several streams, several host threads) race
 * on it and must be serialised by the caller.
 */
PAGED_ATTN_API int paged_attn_decode_static(const void* q, const void* k_cache, const void* v_cache, void* out,
                             const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                             int H_q, int H_kv, int head_dim, int max_blocks_per_seq,
                             int block_size, float scale, void* stream);

/*
 * Device-side checks for every later call of the calling thread: with
 * num_blocks > 0, every decode and append entry point validates the block ids
 * it uses against [0, num_blocks) and reports into *d_status (a device int32,
 * 4-byte aligned, that the caller zero-fills) as paged_attn_decode_checked
 * does: bit 0 for a bad block id (a decode reads zero rows for it through the
 * tensor copies of the standard and FP8 layouts, block 0's rows through the
 * bulk copies of the x-packed layout; an append skips that row), bit 1 for a
 * bad length or a multi-token sequence with more query rows than the call
 * allows, bits 2 and 3 as there.  (0, NULL) turns the checks off.  Returns
 * PAGED_ATTN_ERR_SIZES for num_blocks outside [1, 2^31) and
 * PAGED_ATTN_ERR_POINTER for a null or misaligned d_status, changing nothing.
 */
PAGED_ATTN_API int paged_attn_set_checks(long long num_blocks, int32_t* d_status);

/*
 * The same operation over FP8 caches: the nvfp4-megamoe README's FP8 KV path
 * ("Stage D: FP8 Paged KV Gather", "FP8 KV Quantize/Dequant": e4m3 values,
 * dequantized with a scale per position during the gather).  k_cache / v_cache
 * hold e4m3 bytes (OCP E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities) in the bf16 layout above, 1 byte per element, and
 *   k_scale, v_scale  [num_blocks, H_kv, block_size]  float32  (read)
 * give each cache row its dequant factor:
 *   K_t[d] = e4m3(k_cache[b, g, slot, d]) * k_scale[b, g, slot]   (V alike).
 * head_dim must be 128 or 256 (PAGED_ATTN_ERR_HEAD_DIM otherwise).  The
 * products run on f16 tensor cores: q is rounded to f16 (exact for bf16 values
 * of magnitude 2^-14 .. 65504), the probabilities times the V row factors are
 * rounded to f16; accumulation is fp32.  The probabilities are taken against a
 * running maximum that may trail the true one by up to a factor of 16 (so each
 * is at most 16): V row factors below 4094 (rows of magnitude below about
 * 1.8e6) keep the f16 products finite.  Workspace, allocation and errors as
 * paged_attn_decode; rows past a sequence's length may hold anything (NaN
 * bytes and factors included).
 */
PAGED_ATTN_API int paged_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                                         const float* k_scale, const float* v_scale, void* out,
                                         const int32_t* block_tables, const int32_t* seq_lens,
                                         int num_seqs, int H_q, int H_kv, int head_dim,
                                         int max_blocks_per_seq, int block_size, float scale,
                                         void* stream);

/*
 * Multi-token decode: several new tokens per sequence query the cache at once
 * (speculative decoding, chunked prefill), the ragged query batch of AstrAI's
 * CUDA Kernels page ("Q Scheduling and KV Addressing": rows located through
 * qo_indptr; "Python Wrappers": is_causal).  Sequence s owns the query rows
 * qo_indptr[s] .. qo_indptr[s+1] - 1, its last q_len = qo_indptr[s+1] -
 * qo_indptr[s] tokens, which are already in the cache (seq_lens[s] counts
 * them).  Query i of sequence s attends the tokens t <= seq_lens[s] - q_len + i
 * (causal: its own position and everything before):
 *
 *   out[qo[s] + i, h, :] = softmax_t(scale * q[qo[s] + i, h, :] . K_t) . V_t,
 *                          t in [0, seq_lens[s] - q_len + i]
 *
 *   q, out      [total_q, H_q, head_dim]  bf16 (read / written)
 *   qo_indptr   [num_seqs + 1]  int32, device, 16-byte aligned: qo_indptr[0] = 0,
 *               non-decreasing, qo_indptr[num_seqs] = total_q
 *   max_q_len   the largest q_len (host value); max_q_len * (H_q / H_kv) <= 256
 *
 * Caches, tables, lengths, head_dim, block_size and scale as paged_attn_decode
 * (bf16 caches in the standard layout).  The q_len * G query rows of one KV
 * head are processed together, in pieces of 16 rows when they are more than 8:
 * every piece streams the KV head's pages once.  Rows whose query sees no token
 * (q_len > seq_len) and the rows of empty sequences are zero.  Query rows a
 * sequence does not own are not written.  Returns PAGED_ATTN_ERR_SIZES for
 * total_q < 0, max_q_len < 1 or max_q_len * G > 256; errors otherwise as
 * paged_attn_decode.  Uses the library-owned workspace.
 */
PAGED_ATTN_API int paged_attn_decode_multi(const void* q, const void* k_cache,
                                           const void* v_cache, void* out,
                                           const int32_t* qo_indptr,
                                           const int32_t* block_tables,
                                           const int32_t* seq_lens, int num_seqs, int total_q,
                                           int max_q_len, int H_q, int H_kv, int head_dim,
                                           int max_blocks_per_seq, int block_size, float scale,
                                           void* stream);

/*
 * paged_attn_decode_multi with the causal mask chosen by the caller (AstrAI's
 * CUDA Kernels page, "Python Wrappers": is_causal).  is_causal != 0 is
 * paged_attn_decode_multi; is_causal = 0 lets every query row of sequence s
 * attend all its tokens t < seq_lens[s]:
 *
 *   out[qo[s] + i, h, :] = softmax_t(scale * q[qo[s] + i, h, :] . K_t) . V_t,
 *                          t in [0, seq_lens[s])
 *
 * Everything else as paged_attn_decode_multi.
 */
PAGED_ATTN_API int paged_attn_decode_multi_ex(const void* q, const void* k_cache,
                                              const void* v_cache, void* out,
                                              const int32_t* qo_indptr,
                                              const int32_t* block_tables,
                                              const int32_t* seq_lens, int num_seqs,
                                              int total_q, int max_q_len, int H_q, int H_kv,
                                              int head_dim, int max_blocks_per_seq,
                                              int block_size, float scale, int is_causal,
                                              void* stream);

/*
 * The same operation over bf16 caches in the x-packed layout ("Paged Attention
 * Kernel Architecture for BI-V100", section 3, Paged K/V Gather: the key cache
 * split into 16-byte packs of x = 8 elements, the value cache head_dim-major):
 *
 *   k_cache  [num_blocks, H_kv, head_dim / 8, block_size, 8]  bf16  (read)
 *   v_cache  [num_blocks, H_kv, head_dim, block_size]         bf16  (read)
 *
 * so K_t[d] = k_cache[b, g, d / 8, t % block_size, d % 8] and
 * V_t[d] = v_cache[b, g, d, t % block_size] with b = block_tables[s, t / block_size].
 * Everything else (q, out, tables, lengths, sizes, scale, workspace, errors,
 * rows past a sequence's length) is as paged_attn_decode; the arithmetic is
 * the same, so the output equals paged_attn_decode's over the same values.
 */
PAGED_ATTN_API int paged_attn_decode_xpacked(const void* q, const void* k_cache,
                                             const void* v_cache, void* out,
                                             const int32_t* block_tables,
                                             const int32_t* seq_lens, int num_seqs, int H_q,
                                             int H_kv, int head_dim, int max_blocks_per_seq,
                                             int block_size, float scale, void* stream);

/*
 * Cache append ("reshape and cache") of one new token per sequence, the write
 * that precedes the decode: the paged-decode layout above counts the new token
 * in seq_lens ("context length including the new token"), so its K and V must
 * be in the cache when the decode runs; AstrAI's CUDA-kernels page (Backend
 * Layer) has the backend own that write.  For every sequence s with
 * L = seq_lens[s] >= 1 and every KV head g, with t = L - 1:
 *
 *   k_cache[block_tables[s, t / block_size], g, t % block_size, :] = k_new[s, g, :]
 *   v_cache[...same place...]                                      = v_new[s, g, :]
 *
 *   k_new, v_new  [num_seqs, H_kv, head_dim]  bf16  (read; device, 16-byte aligned)
 *   k_cache, v_cache                          bf16  (written at those rows only)
 *
 * Sequences with L = 0 or L > max_blocks_per_seq * block_size write nothing.
 * The block ids are not checked.  Sizes follow paged_attn_decode's rules
 * (head_dim 64/128/256, block_size 16/32); errors as above.  Asynchronous on
 * `stream`; allocates nothing.
 */
PAGED_ATTN_API int paged_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const int32_t* block_tables,
                                   const int32_t* seq_lens, int num_seqs, int H_kv, int head_dim,
                                   int max_blocks_per_seq, int block_size, void* stream);

/*
 * paged_kv_append followed by paged_attn_decode, fused into the decode launch:
 * the warp that processes the page holding a sequence's new token puts that
 * token's K and V rows into its copy of the page in shared memory (whatever
 * the cache held there is not used) and stores them to the cache, so the
 * append costs no extra launch and no extra pass over the cache.  The blocks
 * that receive the new tokens must not also be read by another sequence of
 * the same call (no copy-on-write sharing of a partly filled block).  When the
 * batch has many (sequence, KV head) pairs per SM (four or more per CTA of the
 * persistent grid), the per-piece patch would sit on the critical path of the
 * CTA crossing the most short sequences, and the call instead runs the append
 * as its own launch just ahead of the decode; the result is the same.  Same
 * arguments, workspace and errors as paged_attn_decode, plus k_new / v_new
 * ([num_seqs, H_kv, head_dim] bf16, 16-byte aligned).
 */
PAGED_ATTN_API int paged_attn_append_decode(const void* q, const void* k_new, const void* v_new,
                                            void* k_cache, void* v_cache, void* out,
                                            const int32_t* block_tables, const int32_t* seq_lens,
                                            int num_seqs, int H_q, int H_kv, int head_dim,
                                            int max_blocks_per_seq, int block_size, float scale,
                                            void* stream);

/*
 * Cache append of several new tokens per sequence, the write that precedes the
 * multi-token decode: the rows of k_new / v_new ([total_q, H_kv, head_dim]
 * bf16, 16-byte aligned) follow qo_indptr as the queries do (AstrAI's CUDA
 * Kernels page, "Q Scheduling and KV Addressing"): row qo_indptr[s] + i is
 * token t = seq_lens[s] - q_len + i of sequence s (q_len = qo_indptr[s+1] -
 * qo_indptr[s]; seq_lens counts the new tokens), and for every KV head g
 *
 *   k_cache[block_tables[s, t / block_size], g, t % block_size, :] = k_new[qo_indptr[s] + i, g, :]
 *
 * (v alike).  Rows with t < 0 (more new rows than the sequence holds), of a
 * sequence with a length outside [1, max_blocks_per_seq * block_size], or
 * outside [qo_indptr[0], qo_indptr[num_seqs]) write nothing.  Sizes and errors
 * as paged_kv_append, plus PAGED_ATTN_ERR_SIZES for total_q < 0.
 * Asynchronous on `stream`; allocates nothing.
 */
PAGED_ATTN_API int paged_kv_append_multi(const void* k_new, const void* v_new, void* k_cache,
                                         void* v_cache, const int32_t* qo_indptr,
                                         const int32_t* block_tables, const int32_t* seq_lens,
                                         int num_seqs, int total_q, int H_kv, int head_dim,
                                         int max_blocks_per_seq, int block_size, void* stream);

/*
 * paged_kv_append_multi followed by paged_attn_decode_multi_ex, as two
 * launches on `stream` (the decode waits for the append to complete before it
 * reads anything, whatever the launch flags).  Arguments as the two calls.
 */
PAGED_ATTN_API int paged_attn_append_decode_multi(const void* q, const void* k_new,
                                                  const void* v_new, void* k_cache,
                                                  void* v_cache, void* out,
                                                  const int32_t* qo_indptr,
                                                  const int32_t* block_tables,
                                                  const int32_t* seq_lens, int num_seqs,
                                                  int total_q, int max_q_len, int H_q, int H_kv,
                                                  int head_dim, int max_blocks_per_seq,
                                                  int block_size, float scale, int is_causal,
                                                  void* stream);

/*
 * Cache append into FP8 caches (quantize on write; nvfp4-megamoe README, "FP8
 * KV Quantize/Dequant" and "Paged KV cache read/write"): the new token's K and
 * V rows of every sequence and KV head, bf16 [num_seqs, H_kv, head_dim], are
 * quantized one row at a time and written where paged_kv_append writes:
 *
 *   f        = max_d |x[d]| / 448   in float32 (f = 1 for an all-zero row)
 *   byte[d]  = e4m3(x[d] / f)       float32 quotient, rounded to nearest even,
 *                                   saturated to +-448
 *   k_cache[b, g, slot, :] = byte,  k_scale[b, g, slot] = f   (v alike)
 *
 * so that paged_attn_decode_fp8 reads x[d] as e4m3(byte[d]) * f.  k_cache /
 * v_cache hold e4m3 bytes, k_scale / v_scale float32 [num_blocks, H_kv,
 * block_size]; head_dim 128 or 256 (PAGED_ATTN_ERR_HEAD_DIM otherwise).
 * Which sequences write, sizes, errors: as paged_kv_append.  Asynchronous on
 * `stream`; allocates nothing.
 */
PAGED_ATTN_API int paged_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, float* k_scale, float* v_scale,
                                       const int32_t* block_tables, const int32_t* seq_lens,
                                       int num_seqs, int H_kv, int head_dim,
                                       int max_blocks_per_seq, int block_size, void* stream);

/*
 * paged_kv_append_fp8 followed by paged_attn_decode_fp8, fused into the decode
 * launch as paged_attn_append_decode is for bf16 caches: the warp that reads the
 * page holding a sequence's new token quantizes the new K and V rows exactly as
 * paged_kv_append_fp8 does, puts the bytes and row floats into its copy of the
 * page in shared memory and stores them to the cache.  For head_dim 256, or
 * with four or more (sequence, KV head) pairs per CTA of the persistent grid,
 * the append runs as its own launch and the decode after it is a plain launch
 * (whatever the launch flags).  The same bytes, floats and output either way.  Arguments as the two
 * calls; the blocks receiving new tokens must not also be read by another
 * sequence of the same call.
 */
PAGED_ATTN_API int paged_attn_append_decode_fp8(const void* q, const void* k_new,
                                                const void* v_new, void* k_cache, void* v_cache,
                                                float* k_scale, float* v_scale, void* out,
                                                const int32_t* block_tables,
                                                const int32_t* seq_lens, int num_seqs, int H_q,
                                                int H_kv, int head_dim, int max_blocks_per_seq,
                                                int block_size, float scale, void* stream);

/* Human-readable text for a PAGED_ATTN_* code (static storage). */
PAGED_ATTN_API const char* paged_attn_status_string(int status);

/*
 * Launch flags for the decode calls made afterwards from the calling host
 * thread (all entry points; 0, the default, restores the plain behaviour).
 * Returns PAGED_ATTN_ERR_FLAGS, and changes nothing, for unknown bits.
 *
 * PAGED_ATTN_FLAG_EARLY_PROLOGUE: every decode launch waits for the work
 * ahead of it in the stream (programmatic dependent launch) before touching
 * global memory.  With this flag the caller guarantees that this earlier work,
 * which may still be running, writes none of k_cache, v_cache (and their row
 * floats), block_tables, seq_lens or qo_indptr.  Only q, the new K/V rows of
 * the fused append and the output may be written by it.  The kernel then
 * scans the lengths, translates the first pages and starts their tensor
 * copies while that work finishes.  It waits for it only before reading q or
 * the new rows, and before writing the output, the workspace or a status
 * word.  In a layer-by-layer decode loop the kernel just before attention
 * typically writes q, and with paged_attn_append_decode the new K/V rows too,
 * but not the caches, tables or lengths.  With the caller's own
 * paged_kv_append (or any other write of the caches) just before, the flag
 * must stay off.  The append-and-decode entry points never let their own
 * append break the guarantee: where the append is a launch of its own, the
 * decode after it is a plain launch whatever the flag says.  Results are
 * those of the plain launch.
 */
PAGED_ATTN_API int paged_attn_set_launch_flags(int flags);

/*
 * Zero-fills the library-owned workspace of the current device on `stream`
 * (nothing to do when none exists yet).  Needed only after a call reported a
 * combine wait that ran out (status bit 2), which can leave split counters set.
 */
PAGED_ATTN_API int paged_attn_reset_workspace(void* stream);

/* The last cudaError_t / CUresult value behind a PAGED_ATTN_ERR_CUDA on this thread. */
PAGED_ATTN_API int paged_attn_last_cuda_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
PAGED_ATTN_API int paged_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */
