/*
 * oracle.h -- CPU oracle for the int8 gradient-bucket quantise + W-way reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded restatement of
 * what the data-parallel gradient-synchronisation path computes.  Only the test
 * suite, the smoke check in __graft_entry__ and the `cpu_baseline` / reference
 * legs of bench.py may load it.  It shares no code, header, table or helper with
 * the CUDA library in dp_gradient_bucket_gb300/, and it includes nothing from it.
 *
 * Sources (pages are named by subject and host):
 *   [HCCL-PIPE]  "pipelined HCCL AllReduce" article, bjdmk.com.cn/news/6235379
 *                §2.1 (dynamic_chunk), §2.2.1 (quantize_gradient, INT8_ALLREDUCE),
 *                §3.1 (per-chunk all_reduce_async), §6.1 (unscale before quantise)
 *   [TITAN-3D]   "torchtitan-npu 3D parallel" article, framerc.cn/news/2545645,
 *                AMP + 3D section (unscale -> fp32 SUM all_reduce -> divide by dp size)
 *   [NPU-DIST]   "torch_npu distributed module" article, hwcomputing.csdn.net,
 *                §2.2 component table (DDP Reducer buckets), §9.2 allreduce_coalesced
 *                (flatten small tensors into one buffer), env-var table (HCCL_DETERMINISTIC)
 *
 * Arithmetic: IEEE-754 binary32, round-to-nearest-even, no contraction (built with
 * -ffp-contract=off), no flush-to-zero.  Every floating-point step is one C++
 * float operation so a reader can check it against the pages by eye.
 *
 * Layout shared with the library (an interface, not code): W virtual-rank rows,
 * row r starting at element r*rank_stride; a chunk table of num_chunks+1 int64
 * element offsets into each row (buckets laid end to end); codes [W][rank_stride]
 * int8; scales [W][num_chunks] float; out [offsets[num_chunks]] float.
 */
#ifndef GQ_ORACLE_H
#define GQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1 };
enum { ORACLE_SEQ = 0, ORACLE_RING = 1, ORACLE_TREE = 2 };

/* dynamic_chunk for one bucket of n elements of eb bytes ([HCCL-PIPE] §2.1):
 * k = max(1, nbytes // (131072 - 131072 % 64)); torch.chunk(bucket, k) splits into
 * pieces of c = ceil(n / k) elements, the last one shorter, ceil(n / c) pieces in all.
 * n == 0 gives one empty chunk (torch.chunk of an empty tensor).
 * Returns the chunk count; *chunk_elems receives c (0 for n == 0). */
int64_t oracle_bucket_chunks(int64_t n, int64_t eb, int64_t* chunk_elems);

/* The same with the base chunk size as a parameter (the page's CHUNK_SIZE; [HCCL-PIPE] §4.2
 * Config knobs, §2.1): k = max(1, nbytes // (chunk_size - chunk_size % 64)). */
int64_t oracle_bucket_chunks_sized(int64_t n, int64_t eb, int64_t chunk_size, int64_t* chunk_elems);

/* Scope of one quantisation scale.  CHUNK: dynamic_chunk pieces of every entry (entries are
 * buckets), with chunk_size as the base size.  BUCKET / TENSOR: each entry (a bucket, or a
 * tensor) is one chunk, so one scale covers it whole -- the page's quantize_gradient applied
 * to the whole gradient it is given ([HCCL-PIPE] §2.2.1), per bucket or per tensor.  An empty
 * entry is one empty chunk.  Entries are laid end to end. */
enum { ORACLE_SCOPE_CHUNK = 0, ORACLE_SCOPE_BUCKET = 1, ORACLE_SCOPE_TENSOR = 2 };

/* Chunk table of count entries under a scope (writes count-dependent num_chunks+1 offsets when
 * capacity >= num_chunks+1).  Returns num_chunks, or -1 on a negative size, an unknown scope or
 * (scope CHUNK) a chunk size whose 64-byte-aligned part is 0. */
int64_t oracle_plan_chunks_ex(const int64_t* elems, int64_t count, int64_t eb, int scope, int64_t chunk_size,
                              int64_t* offsets, int64_t capacity);

/* Chunk table for buckets laid end to end.  Writes num_chunks+1 offsets when
 * capacity >= num_chunks+1 (else writes nothing).  Returns num_chunks, or -1 on a
 * negative size. */
int64_t oracle_plan_chunks(const int64_t* bucket_elems, int64_t num_buckets, int64_t eb,
                           int64_t* offsets, int64_t capacity);

/* DDP-Reducer-style bucket assignment ([NPU-DIST] §2.2 Reducer, §9.2 coalescing):
 * tensors in list order; a tensor goes into the open bucket unless that bucket is
 * non-empty and the tensor would push it past cap_bytes, in which case the bucket
 * is closed and a new one opened.  Writes bucket_of_tensor[t] and bucket_elems[b]
 * (capacity max_buckets).  Returns the bucket count, or -1 if it exceeds capacity. */
int64_t oracle_assign_buckets(const int64_t* tensor_elems, int64_t num_tensors, int64_t eb,
                              int64_t cap_bytes, int64_t* bucket_of_tensor,
                              int64_t* bucket_elems, int64_t max_buckets);

/* quantize_gradient per (rank, chunk) ([HCCL-PIPE] §2.2.1), after the optional
 * unscale ([HCCL-PIPE] §6.1, [TITAN-3D] AMP section):
 *   g = float(x) * inv,  inv = (float)(1.0 / (double)loss_scale)
 *   m = max |g|;  s = m / 127.0f;
 *   q = (s == 0) ? 0 : clamp(rint(g / s), -128, 127)    (rint: ties to even)
 * dt: ORACLE_F32 (float rows) or ORACLE_F16 (IEEE binary16 bit patterns).
 * Returns the number of (rank, chunk) pairs that held a non-finite value (their
 * codes and scale are unspecified; codes are written as 0 there). */
int64_t oracle_quantize(const void* grads, int dt, int W, int64_t rank_stride,
                        const int64_t* offsets, int64_t num_chunks, float loss_scale,
                        int8_t* codes, float* scales);

/* INT8_ALLREDUCE arithmetic + mean ([HCCL-PIPE] §2.2.1, §3.1; [TITAN-3D] AMP section):
 * d_r = (float)q_r * s_r;  acc summed over the W ranks in the given order;
 * out = acc / (float)W.
 *   SEQ : ranks 0, 1, ..., W-1
 *   RING: element in segment t of its chunk (torch.chunk(chunk, W)) starts at rank
 *         (t+1) % W and continues (t+2) % W, ..., t
 *   TREE: pairwise over ranks in index order, an odd one carried up a level. */
void oracle_reduce(const int8_t* codes, const float* scales, int W, int64_t rank_stride,
                   const int64_t* offsets, int64_t num_chunks, int order, float* out);

/* The same arithmetic in the hierarchical (topology-aware) order ([HCCL-PIPE] §2.1 third
 * stage: a flat ring over all cards replaced by one ring inside each machine plus an
 * aggregation tree between machines; §3.2 intra-machine groups and inter-machine tree).
 * The W ranks form W / L nodes of L consecutive ranks (node n = ranks n*L .. n*L+L-1).
 * For an element in segment t of torch.chunk(chunk, L), node n sums its ranks in ring
 * order: local rank (t+1) % L first, then (t+2) % L, ..., t.  The W / L node sums are then
 * added pairwise in node index order, an odd one carried up a level (the TREE rule over
 * nodes); out = acc / (float)W.  L == W is the RING order and L == 1 the TREE order.
 * Returns 0, or -1 (writing nothing) if L < 1 or W % L != 0. */
int oracle_reduce_hier(const int8_t* codes, const float* scales, int W, int64_t rank_stride,
                       const int64_t* offsets, int64_t num_chunks, int L, float* out);

/* One step of the dynamic loss-scale update that follows the found-inf check in a mixed-precision
 * step ([HCCL-PIPE] §6.1 mixed precision; torch.cuda.amp.GradScaler.update semantics):
 *   found_inf != 0 (NaN counts as set): scale = (float)(scale * backoff), tracker = 0
 *   otherwise: t = tracker + 1; if t == interval: g = (float)(scale * growth), scale = g only
 *              if g is finite, tracker = 0; else tracker = t. */
void oracle_amp_update_scale(float* scale, int32_t* tracker, float found_inf, float growth, float backoff,
                             int32_t interval);

/* Exact binary16 -> binary32 decode (used by the oracle's F16 path; exported so the
 * decode can be pinned on its own). */
float oracle_half_to_float(uint16_t h);

#ifdef __cplusplus
}
#endif
#endif
