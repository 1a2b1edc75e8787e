/*
 * ring_attn.h -- C ABI of libringattn.so: blockwise ring attention on one
 * NVIDIA B300 (sm_103a).
 *
 * What is computed.  Ring attention ("Sequenzparallelitaet und
 * Ringaufmerksamkeit", section "Tiefer Einblick"; "Context parallelism and
 * zig-zag ring attention", section "Zig Zag Ring Attention") splits a
 * sequence of S tokens into P shards.  Each shard keeps its queries while the
 * key/value blocks of all shards travel around a ring; at ring step t shard r
 * holds the block of shard s = (r - t) mod P, computes partial attention and
 * folds it into a running maximum and normaliser (online softmax), rescaling
 * the earlier partial sums.  After P steps every query has attended to every
 * key, and the result equals full attention.  On one GPU the P ring ranks are
 * virtual shards: the ring is a block schedule, no bytes cross a GPU boundary.
 *
 * Shard layouts (which tokens a shard owns; n = S / P, C = S / (2P)):
 *   RA_LAYOUT_CONTIGUOUS  shard r owns tokens [r*n, (r+1)*n)  ("Tiefer Einblick").
 *   RA_LAYOUT_STRIPED     token i belongs to shard i mod P  (the interleaving
 *                         shown in "Zig Zag Ring Attention": GPU 0 gets tokens
 *                         0, 4, 8, ..., GPU 1 gets 1, 5, 9, ...; that page
 *                         calls it zig-zag).
 *   RA_LAYOUT_ZIGZAG      cut into 2P chunks of C tokens; shard r owns chunks r
 *                         and 2P-1-r (the variant named in "Die Zukunft der
 *                         Sequenzparallelitaet"; the pages give no definition,
 *                         this is the reading this library implements).
 * Inside a shard, tokens keep increasing global position ("local slot" j).
 * The causal mask always compares GLOBAL positions: query i sees key j iff
 * j <= i ("Zig Zag Ring Attention": an autoregressive token only sees earlier
 * tokens).
 *
 * Tensors (row-major, caller-allocated, device memory unless stated):
 *   q, out, dout, dq   [B][S][H][D]    natural token order
 *   k, v, dk, dv       [B][S][Hkv][D]  natural token order
 *   lse                [B][H][S]       fp32, natural log-sum-exp of the scaled
 *                                      scores (lse = m + ln l)
 *   q_shard, out_part  [B][n][H][D]    one shard, local-slot order
 *   k_shard, v_shard   [B][n][Hkv][D]  one shard, local-slot order
 *   lse_part           [B][H][n]       fp32
 * bf16 unless stated.  Query head h reads key/value head h / (H / Hkv).
 * D must be 64 or 128.  Every pointer must be 16-byte aligned.
 *
 * Ownership and ordering.  The caller owns every buffer; the library keeps no
 * pointer after a call returns.  Every call is asynchronous and ordered on
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 * Transient workspace, when a call needs one, is taken with cudaMallocAsync
 * and released with cudaFreeAsync on that stream.  Calls on different streams
 * may run concurrently.
 *
 * Errors.  Argument errors are detected on the host before anything is
 * launched and return a nonzero ra_status; ring_attn_last_error() then gives
 * a message (per host thread).  A failed launch returns RA_ERR_CUDA.  Kernel
 * waits are bounded in time: a pipeline that stops making progress gives up
 * after about two seconds and leaves a code that ring_attn_check_status()
 * reports as RA_ERR_DEVICE_TIMEOUT.
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_NULL = 1,           /* a required pointer is NULL */
  RA_ERR_SHAPE = 2,          /* sizes inconsistent or out of range */
  RA_ERR_LAYOUT = 3,         /* unknown layout, or S not divisible as it needs */
  RA_ERR_UNSUPPORTED = 4,    /* D not 64/128, non-finite scale, no sm_100-class GPU */
  RA_ERR_ALIGN = 5,          /* a pointer is not 16-byte aligned */
  RA_ERR_CUDA = 6,           /* a CUDA runtime call or launch failed */
  RA_ERR_DEVICE_TIMEOUT = 7, /* a kernel gave up waiting (see ring_attn_check_status) */
  RA_ERR_ALLOC = 8           /* workspace allocation failed */
} ra_status;

typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0,
  RA_LAYOUT_STRIPED = 1,
  RA_LAYOUT_ZIGZAG = 2
} ra_layout;

typedef enum { RA_BF16 = 0, RA_F32 = 1 } ra_dtype;

/*
 * ring_attn_fwd -- the whole ring: for every shard r, steps t = 0..P-1 over
 * blocks s = (r - t) mod P, online-softmax accumulation, final normalisation.
 * ("Tiefer Einblick": after one full loop every query has attended to every
 * key.)  Equal to softmax(scale * q k^T + causal mask) v.
 *   out:  [B][S][H][D], bf16 (out_dtype RA_BF16) or fp32 (RA_F32).
 *   lse:  [B][H][S] fp32 (may be NULL if not wanted).
 *   scale: multiplies q.k before the softmax (usually 1/sqrt(D)); finite.
 * Needs S % P == 0 (and S % 2P == 0 for zig-zag), H % Hkv == 0, S >= 1.
 * Key blocks that the causal mask hides entirely are skipped, never computed.
 */
ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out,
                        ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int64_t S,
                        int D, int P, ra_layout layout, int causal, float scale,
                        void* stream);

/*
 * ring_attn_fwd_varlen -- ring_attn_fwd over packed sequences: nseq sequences
 * of different lengths laid end to end, each one split over the P ranks by
 * `layout` on its own and attending only within itself.  This is the next step
 * the pages point to beyond one sequence: sequence parallelism for long
 * documents and code bases in training and inference ("Die Zukunft ..." and
 * its use cases); the packing itself is this library's reading.
 *   cu_seqlens: HOST array of nseq+1 int64 token offsets, cu_seqlens[0] = 0,
 *               sequence i holds tokens [cu_seqlens[i], cu_seqlens[i+1]);
 *               every length must be divisible by P (by 2P for zig-zag).
 *   q, out [total][H][D]; k, v [total][Hkv][D] (total = cu_seqlens[nseq]);
 *   lse [H][total] fp32 or NULL.  Other rules as ring_attn_fwd.
 * The call copies a work list (longest first) and cu_seqlens to the device
 * with cudaMallocAsync / cudaMemcpyAsync / cudaFreeAsync on `stream`.
 */
ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                               ra_dtype out_dtype, float* lse, const int64_t* cu_seqlens, int nseq,
                               int H, int Hkv, int D, int P, ra_layout layout, int causal,
                               float scale, void* stream);

/*
 * ring_attn_fwd_counted -- ring_attn_fwd that also adds, for each shard r, the
 * number of (128-query tile, 128-key tile) blocks the kernel actually
 * multiplied into shard_tiles[r] (device, int64[P], caller-zeroed).  The
 * per-shard totals measure the causal load balance the interleaved layouts are
 * meant to fix ("Zig Zag Ring Attention": with contiguous shards the later
 * ranks carry more work and the earlier ones idle).
 */
ra_status ring_attn_fwd_counted(const void* q, const void* k, const void* v, void* out,
                                ra_dtype out_dtype, float* lse, int B, int H, int Hkv,
                                int64_t S, int D, int P, ra_layout layout, int causal,
                                float scale, int64_t* shard_tiles, void* stream);

/*
 * ring_attn_fwd_traced -- ring_attn_fwd that also records a timeline of its
 * work items (a pair of 128-row query tiles of one shard, batch entry and
 * head): records[4*i .. 4*i+3] = the %globaltimer (ns) when a CTA took item i
 * up, when its last output row was stored, (shard << 32) | CTA index, and the
 * number of key tiles its query tiles multiplied.  Grouped by shard, the
 * records show per-rank busy time: the load balance that "Zig Zag Ring
 * Attention" sets out to fix, measured rather than counted.
 *   records: device int64, 8-byte aligned, at least 4 * *items words; the call
 *   clears it on `stream` first.  capacity: records it holds (in items).
 *   items: host int64, receives the number of work items of this call.
 */
ra_status ring_attn_fwd_traced(const void* q, const void* k, const void* v, void* out,
                               ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int64_t S,
                               int D, int P, ra_layout layout, int causal, float scale,
                               int64_t* records, int64_t capacity, int64_t* items, void* stream);

/*
 * ring_attn_bwd -- gradients of ring_attn_fwd (the pages describe the forward
 * only; this is the standard softmax-attention gradient):
 *   P = exp(scale q k^T - lse), delta = rowsum(dout * out),
 *   dv = P^T dout, dS = P * (dout v^T - delta), dq = scale dS k, dk = scale dS^T q,
 * with dk, dv summed over the H/Hkv query heads sharing a key/value head.
 *   out, lse: the forward's outputs (out bf16, lse [B][H][S] fp32).
 *   dout: [B][S][H][D] bf16.  dq [B][S][H][D], dk/dv [B][S][Hkv][D]: bf16 outputs,
 *   every element written.
 * Same size, layout and scale rules as ring_attn_fwd (out_dtype bf16 only).
 * The key/value blocks meet the query shards in ring order; dq is computed in
 * a separate pass over the query tiles, so no atomics are used and the
 * result is deterministic.  Takes a transient fp32 workspace of
 * 8 * B * H * P * T * 128 bytes (T = 128-slot tiles per shard, counted per
 * zig-zag chunk) with cudaMallocAsync / cudaFreeAsync on `stream`; returns
 * RA_ERR_ALLOC if that fails.
 */
ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H, int Hkv, int64_t S, int D, int P, ra_layout layout,
                        int causal, float scale, void* stream);

/*
 * ring_attn_bwd_varlen -- gradients of ring_attn_fwd_varlen (packed
 * sequences; same cu_seqlens, layouts and shapes):
 *   q, out, dout, dq [total][H][D]; k, v, dk, dv [total][Hkv][D];
 *   lse [H][total] fp32 from ring_attn_fwd_varlen (out bf16).
 * Each sequence's gradients are those of its own attention.  Takes a
 * transient workspace (vectors and work lists) with cudaMallocAsync /
 * cudaMemcpyAsync / cudaFreeAsync on `stream`.
 */
ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               const int64_t* cu_seqlens, int nseq, int H, int Hkv, int D, int P,
                               ra_layout layout, int causal, float scale, void* stream);

/*
 * ring_attn_bwd_noalloc -- ring_attn_bwd for callers that cannot allocate GPU
 * memory while they run: a framework that has already reserved the whole
 * device for its own caching allocator (so a driver allocation from inside
 * a library fails or fragments that pool), or a program whose policy forbids
 * allocation after start-up.  The pages have no counterpart of this call; it
 * only changes where the backward's scratch lives.
 *   Arguments, layouts, results and checks are those of ring_attn_bwd.  The
 *   caller still passes every input and output.
 *   The scratch (-lse*log2(e) and -delta in tile order) is a 16 MiB array that
 *   the library reserves statically on every GPU that loads it, held until
 *   the process exits.  Limit: B * H * P * T * 128 <= 2097152 (T = 128-slot
 *   tiles per shard, counted per zig-zag chunk); larger problems get
 *   RA_ERR_SHAPE with a message, and should use ring_attn_bwd.
 *   No cudaMalloc, cudaMallocAsync, cudaFree or other allocating call is made.
 *   Each call outside stream capture looks up the array's device address with
 *   the current device (so a device reset that reloads the library's module is
 *   followed); a call made while `stream` is capturing reuses the address the
 *   last uncaptured call found on that device.  Make the first call on each
 *   device before any stream capture: a captured first call is refused with
 *   RA_ERR_UNSUPPORTED.
 *   Every call shares the one array and it keeps the last call's contents;
 *   each call writes every scratch element it reads before reading it, so
 *   nothing needs clearing.  Calls whose kernels overlap on the GPU (other
 *   streams, other host threads) race on the array: serialise them.
 */
ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H, int Hkv, int64_t S, int D, int P, ra_layout layout,
                                int causal, float scale, void* stream);

/*
 * ring_attn_decode -- inference step against a sharded key/value cache.  The
 * pages put ring attention to work on ultra-long-context inference
 * ("Sequenzparallelitaet und Ringaufmerksamkeit", "Die Zukunft ..." and its
 * use cases), with the history's keys and values kept in a cache and read
 * back rather than recomputed (the Chinese article on long-context
 * inference).  T new query tokens at positions S-T .. S-1 attend to the S
 * cached tokens (their own keys and values already appended): query t sees
 * the keys at positions <= S-T+t.  The P ranks of the ring hold the cache by
 * `layout`; each computes a partial over the keys it holds, and the partials
 * are merged as in ring_attn_merge.  Equal to ring_attn_fwd's rows S-T .. S-1.
 *   q        [B][T][H][D] bf16
 *   k_cache, v_cache  [B][S][Hkv][D] bf16, natural token order
 *   out      [B][T][H][D], bf16 (RA_BF16) or fp32 (RA_F32)
 *   lse      [B][H][T] fp32, or NULL
 * Needs (H/Hkv) * T <= 4096 and 1 <= T <= S, plus ring_attn_fwd's size rules;
 * each group of 16 of a kv head's query rows runs as its own CTA over the
 * same cache chunk (T > 1 covers a chunked prefill or a verify step).
 * The step reads the whole cache once: it is bound by HBM bandwidth and runs
 * on the CUDA cores.  Takes a transient fp32 workspace for the partials with
 * cudaMallocAsync / cudaFreeAsync on `stream`; returns RA_ERR_ALLOC if that
 * fails.
 */
ra_status ring_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
                           ra_dtype out_dtype, float* lse, int B, int H, int Hkv, int T, int64_t S,
                           int D, int P, ra_layout layout, float scale, void* stream);

/*
 * ring_attn_cache_append -- writes the keys and values of T new tokens into
 * the cache at positions pos .. pos+T-1: k_cache[b][pos+t] = k_new[b][t] and
 * likewise v, for every kv head.  The Chinese article on long-context
 * inference keeps the history's keys and values in a cache and reads them
 * back instead of recomputing them; this is the write side of that cache,
 * called before ring_attn_decode (whose S is then pos + T).
 *   k_cache, v_cache [B][S_cap][Hkv][D] bf16, natural token order (the
 *   layout's shards are read from it in place);
 *   k_new, v_new [B][T][Hkv][D] bf16.
 * Needs pos + T <= S_cap, D 64 or 128, 16-byte aligned non-overlapping
 * buffers.  A plain copy: the bytes land unchanged.
 */
ra_status ring_attn_cache_append(void* k_cache, void* v_cache, const void* k_new,
                                 const void* v_new, int B, int Hkv, int64_t S_cap, int64_t pos,
                                 int T, int D, void* stream);

/*
 * ring_attn_step -- one ring hop: the queries of shard r against the key/value
 * block of shard s only ("Tiefer Einblick": as each block arrives the GPU
 * computes a partial attention), causal on global positions, normalised
 * within the block.
 *   q_shard [B][n][H][D], k_shard/v_shard [B][n][Hkv][D] (bf16, local order);
 *   out_part [B][n][H][D] fp32, lse_part [B][H][n] fp32.
 * A query that sees no key of the block gets out_part 0 and lse_part -inf.
 */
ra_status ring_attn_step(const void* q_shard, const void* k_shard, const void* v_shard,
                         float* out_part, float* lse_part, int B, int H, int Hkv, int64_t S,
                         int D, int P, ra_layout layout, int r, int s, int causal, float scale,
                         void* stream);

/*
 * ring_attn_step_bwd -- one ring hop of the backward: the queries of shard r
 * against the key/value block of shard s only.  In the pages' ring the
 * key/value blocks travel from rank to rank ("Tiefer Einblick"); the
 * backward of that ring lets each block's dk/dv accumulators travel with it
 * and keeps dq at the queries' rank.  This call computes one hop's share, with
 * lse_shard the FINAL log-sum-exp of shard r's queries (over all blocks, as
 * ring_attn_fwd or a full ring of ring_attn_step/merge produced it):
 *   P = exp(scale q_r k_s^T - lse_r) (causal on global positions),
 *   delta_r = rowsum(dout_r * out_r),  dS = P * (dout_r v_s^T - delta_r),
 *   dq_part (+)= scale dS k_s,  dk_part (+)= scale dS^T q_r,  dv_part (+)= P^T dout_r,
 * dk_part, dv_part summed over the H/Hkv query heads of a key/value head.
 *   q_shard, out_shard, dout_shard [B][n][H][D] bf16 (shard r, local order);
 *   k_shard, v_shard [B][n][Hkv][D] bf16 (block s, local order);
 *   lse_shard [B][H][n] fp32 (shard r);
 *   dq_part [B][n][H][D], dk_part, dv_part [B][n][Hkv][D]: fp32, every element
 *   written (accumulate = 0) or added to (accumulate != 0).
 * Summed over s = 0..P-1 (any order), dq_part is shard r's dq; summed over
 * r, dk_part / dv_part are block s's dk / dv.  Same size rules as
 * ring_attn_fwd; 16-byte aligned pointers.  Takes a transient workspace of
 * 8 * B * H * T * 128 bytes (T = 128-slot tiles of one shard) with
 * cudaMallocAsync / cudaFreeAsync on `stream`.
 */
ra_status ring_attn_step_bwd(const void* q_shard, const void* k_shard, const void* v_shard,
                             const void* out_shard, const float* lse_shard,
                             const void* dout_shard, float* dq_part, float* dk_part,
                             float* dv_part, int B, int H, int Hkv, int64_t S, int D, int P,
                             ra_layout layout, int r, int s, int causal, float scale,
                             int accumulate, void* stream);

/*
 * ring_attn_merge -- fold one partial into a running result, the online
 * softmax accumulation across hops ("Tiefer Einblick"; "technical insight"
 * of the Thai edition: keep a running maximum and normaliser and rescale the
 * earlier partial sums).  With lse = ln(e^lse_acc + e^lse_part):
 *   out_acc = e^(lse_acc - lse) out_acc + e^(lse_part - lse) out_part,
 *   lse_acc = lse.
 * out_* [B][n][H][D] fp32, lse_* [B][H][n] fp32; in place on (out_acc, lse_acc).
 * A -inf lse on one side leaves the other unchanged; both -inf gives (0, -inf).
 */
ra_status ring_attn_merge(float* out_acc, float* lse_acc, const float* out_part,
                          const float* lse_part, int B, int H, int64_t n, int D, void* stream);

/*
 * ring_attn_permute -- move token rows between natural order and shard-major
 * order: dst[o][r*n + j] = src[o][pos_r(j)] (inverse = 0), or the reverse
 * scatter (inverse != 0), for o < outer, where pos_r(j) is the global position
 * held in local slot j of shard r under `layout`.  row_bytes is the size of
 * one token row (H*D*2 for a bf16 [B][S][H][D] tensor with outer = B; 4 for an
 * lse tensor with outer = B*H) and must be a multiple of 4.  src and dst must
 * not overlap.
 */
ra_status ring_attn_permute(const void* src, void* dst, int64_t outer, int64_t S,
                            int64_t row_bytes, int P, ra_layout layout, int inverse,
                            void* stream);

/*
 * ring_attn_permute_shards -- the same row permutation with the shard
 * outermost: dst[r][o][j] = src[o][pos_r(j)] (inverse = 0), or the scatter
 * back (inverse != 0), for o < outer.  Each shard's rows form one contiguous
 * block of outer * n rows: the block an all-to-all sends to (or received from)
 * rank r.  Used by the head-sharded scheme the SP/EP page names beside Ring
 * Attention (Ulysses), whose all-to-all trades a sequence shard of every head
 * for the whole sequence of a head group.  Sizes, alignment and overlap rules
 * as ring_attn_permute; S < 2^31.
 */
ra_status ring_attn_permute_shards(const void* src, void* dst, int64_t outer, int64_t S,
                                   int64_t row_bytes, int P, ra_layout layout, int inverse,
                                   void* stream);

/*
 * ring_attn_head_split -- dst[p][row] = src[row][p] (inverse = 0) or
 * dst[row][p] = src[p][row] (inverse != 0) for `rows` rows of `parts` chunks of
 * chunk_bytes each.  A [B][n][H][D] tensor (rows = B*n, chunk = H/parts heads)
 * becomes one block per head group, the block the head-sharded all-to-all
 * sends to rank p; an lse [B][H][n] (rows = B, chunk = (H/parts)*n*4 bytes)
 * likewise.  chunk_bytes a multiple of 4; 4-byte aligned, non-overlapping
 * buffers (16-byte alignment and chunk sizes take the vector path).
 */
ra_status ring_attn_head_split(const void* src, void* dst, int64_t rows, int parts,
                               int64_t chunk_bytes, int inverse, void* stream);

/*
 * ring_attn_finalize -- out[i] = bf16(acc[i]) for count fp32 values (count a
 * multiple of 4; acc 16-byte and out 8-byte aligned): a rank's fp32 ring
 * accumulator, after the last block has been folded in with ring_attn_merge,
 * stored in the output type (the final store of the forward).
 */
ra_status ring_attn_finalize(const float* acc, void* out, int64_t count, void* stream);

/*
 * ring_attn_index_map -- host-side layout map: pos[r*n + j] = global position
 * of local slot j of shard r (host array of S int64).  No GPU involved.
 */
ra_status ring_attn_index_map(int64_t S, int P, ra_layout layout, int64_t* pos);

/*
 * ring_attn_census -- host-side per-shard work accounting under the kernels'
 * tiling (128-slot tiles that never straddle a contiguous run of positions):
 * visible_pairs[r] = number of (query, key) pairs the mask lets shard r's
 * queries see; computed_tiles[r] = number of (query tile, key tile) blocks
 * the forward kernel multiplies for shard r.  Either pointer may be NULL.
 */
ra_status ring_attn_census(int64_t S, int P, ra_layout layout, int causal,
                           int64_t* visible_pairs, int64_t* computed_tiles);

/*
 * ring_attn_work_schedule -- host side, no GPU involved: the list of work
 * items each CTA of a persistent kernel of a ring-mode call of this shape
 * takes, for a GPU of `sms` SMs and l2_bytes of L2.  kind 0: the forward
 * (a work item is a pair of 128-row query tiles of one (b, head)); 1: the
 * backward's dK/dV pass (one 128-key tile of one (b, kv head)); 2: its dQ pass
 * (one 128-row query tile of one (b, head)).  The item list of each kernel is
 * ordered so that CTAs running at the same time share tiles in L2, longest
 * first within a group; the schedule hands the items out in that order, each
 * to the CTA whose items so far sum to the least estimated work (tiles
 * multiplied, plus a fixed cost per item), as a queue would when CTAs fall
 * idle.  Work is the same whichever CTA takes an item, so the results do not
 * depend on the schedule.  It is a scheduling policy of this library, with no
 * counterpart on the pages.  The calls that launch these kernels build it on
 * the first call of a shape (outside stream capture), copy it to device memory
 * synchronously and keep it for the life of the process, up to 64 MiB of
 * schedules in all; shapes past that, and ring_attn_bwd_noalloc, run without
 * one.
 *
 * Layout (int32): offsets[G + 1] (G = the grid, min(items, sms)), then CTA 0's
 * item ids in the order it takes them, CTA 1's, ...; CTA c's are the entries
 * offsets[c] .. offsets[c+1]-1 after the offsets.  *n_out receives the number
 * of ints, 0 when the call runs without a schedule (no more items than CTAs,
 * or more than 2^22 items; each CTA c then takes item k*G + c in even rounds
 * k and k*G + G-1-c in odd ones).  out == NULL only sizes it; otherwise
 * capacity ints must hold it (RA_ERR_SHAPE if not).  Shape errors as
 * ring_attn_fwd.
 */
ra_status ring_attn_work_schedule(int kind, int B, int H, int Hkv, int64_t S, int D, int P,
                                  ra_layout layout, int causal, int sms, int64_t l2_bytes,
                                  int* out, int64_t capacity, int64_t* n_out);

/*
 * ring_attn_check_status -- waits for `stream`, then reports and clears the
 * device status word: RA_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded
 * wait since the last check, RA_ERR_CUDA if the stream holds an error, else RA_OK.
 */
ra_status ring_attn_check_status(void* stream);

/*
 * ring_attn_wait_selfcheck -- exercises the failure path every kernel's waits
 * share, without a fault: one thread waits on a barrier that nothing ever
 * completes, gives up after limit_ms (1..1000) milliseconds, records a timeout
 * in the device status word and returns; the context stays usable.  The next
 * ring_attn_check_status() then reports RA_ERR_DEVICE_TIMEOUT and clears it.
 * waited_ns (device, int64, 8-byte aligned) receives the time the wait took.
 * The pages have no counterpart of this call (they ask only that failures be
 * tested).
 */
ra_status ring_attn_wait_selfcheck(int limit_ms, int64_t* waited_ns, void* stream);

/*
 * ring_attn_set_wait_limit -- the time limit of every kernel's bounded waits
 * on the current device, in nanoseconds; 0 restores the default (about two
 * seconds).  Tests of the failure path set a limit so short that the waits of
 * an ordinary call run out: the kernels then give up, wait for their own
 * copies and products still in flight, free their tensor memory and return,
 * and ring_attn_check_status() reports RA_ERR_DEVICE_TIMEOUT.  Synchronous;
 * make no call on another stream meanwhile.  The pages have no counterpart
 * (they ask only that failures be detected and tested).
 */
ra_status ring_attn_set_wait_limit(int64_t limit_ns);

/* ring_attn_last_error -- message for the last failing call on this host thread. */
const char* ring_attn_last_error(void);

/* ring_attn_version -- library version string. */
const char* ring_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
