/*
 * ringattn.h -- C ABI of libringattn.so: ring-order (context-parallel)
 * attention, its zigzag token partition, the LSE merge and the
 * context-parallel KV-cache decode path, on one GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every function returns ra_status; nothing is thrown across the ABI.
 *   On failure ra_last_error() (thread-local) describes the first problem.
 * - Arguments are validated on the host before anything is launched: an
 *   invalid argument launches nothing.
 * - The caller owns every buffer.  The library never allocates device
 *   memory; where scratch is needed the caller passes a workspace whose size
 *   a *_workspace_size function reports.
 * - "device" pointers are CUDA global-memory addresses of the current device;
 *   "host" pointers are ordinary CPU memory read during the call.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and is asynchronous: outputs are ready once the stream is.
 * - Kernels never trap.  A bounded device-side wait that expires, or a
 *   device-side bounds check that fails, records a status in a device error
 *   word; ra_device_status() synchronises the stream and returns (and clears)
 *   it.
 * - Tensors are dense and row-major in the layouts stated per function.
 *   Token-major layouts put all heads of a token together: [tokens, H, d].
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ra_stream; /* == cudaStream_t */

typedef enum ra_status {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1, /* bad size, pointer, alignment or rule violation */
  RA_ERR_UNSUPPORTED = 2, /* valid, but not implemented (e.g. head dim)     */
  RA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed              */
  RA_ERR_TIMEOUT = 4,     /* a bounded device wait expired                  */
  RA_ERR_DEVICE_BOUNDS = 5 /* a device-side index check failed (input data) */
} ra_status;

typedef enum ra_dtype { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

/* Token order of the attention tensors.
 * RA_LAYOUT_NATURAL: row of (sequence b, position p) = b*S + p.
 * RA_LAYOUT_ZIGZAG : the gathered head-tail order of ra_zigzag_partition for
 *   B sequences of equal length S: rank-major, then sequence, then the rank's
 *   two chunks (chunk r, then chunk 2N-1-r), each S/(2N) tokens long; the row
 *   of (rank r, sequence b, half h, offset o) is ((r*B + b)*2 + h)*S/(2N) + o.
 *   This is what N context-parallel ranks hold, concatenated. */
typedef enum ra_layout { RA_LAYOUT_NATURAL = 0, RA_LAYOUT_ZIGZAG = 1 } ra_layout;

/* Thread-local description of the last failure ("" if none). */
const char* ra_last_error(void);

/* Library version string. */
const char* ra_version(void);

/* Synchronise `stream`, then return and clear the device error word of every
 * kernel module (RA_OK if no kernel recorded a problem).  A CUDA error seen
 * while synchronising is returned as RA_ERR_CUDA. */
ra_status ra_device_status(ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_zigzag_partition -- head-tail token partition and its restore index.
 * Source: vLLM-Ascend developer guide "Context Parallel (CP)", section
 * "Prefill context parallel (PCP)", head-tail token partition (pad, cut into
 * 2*pcp equal parts, pair part i with part 2*pcp-1-i, pcp_allgather_restore_idx).
 *
 * seq_lens   host   int64 [num_seqs], lengths L_q >= 0 (tokens packed request
 *                   after request, unpadded, in the original order).
 * n_ranks    N >= 1 context-parallel ranks.
 * perm       device int32 [G] out, G = sum_q ceil(L_q/2N)*2N: perm[g] is the
 *                   original token index at gathered position g, -1 for a pad
 *                   position.  Gathered order: rank-major, then request, then
 *                   (chunk r, chunk 2N-1-r) of that request.
 * restore    device int32 [sum L_q] out: restore[i] = gathered position of
 *                   original token i (restore = perm^-1).
 * padded_total, total  host int64 out (may be NULL): G and sum L_q.
 * Either of perm/restore may be NULL to query the sizes only (then nothing is
 * launched).  Errors: num_seqs < 0, n_ranks < 1, negative length, G >= 2^31.
 * ---------------------------------------------------------------------- */
ra_status ra_zigzag_partition(const int64_t* seq_lens, int32_t num_seqs, int32_t n_ranks,
                              int32_t* perm, int32_t* restore, int64_t* padded_total,
                              int64_t* total, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_gather_rows -- dst[i, :] = src[idx[i], :] (a zero row where idx[i] < 0).
 * The data movement of the zigzag permute (idx = perm) and of the restore
 * (idx = restore), same source as ra_zigzag_partition.
 *
 * src  device [src_rows, row_bytes] bytes; idx device int32 [rows];
 * dst  device [rows, row_bytes] out (must not overlap src).
 * An idx >= src_rows is a device-side bounds error (row zero-filled,
 * RA_ERR_DEVICE_BOUNDS recorded).
 * ---------------------------------------------------------------------- */
ra_status ra_gather_rows(const void* src, int64_t src_rows, const int32_t* idx, void* dst,
                         int64_t rows, int64_t row_bytes, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_rope_gather -- rotary position embedding of Q or K rows, fused with the
 * row gather of the zigzag permute:
 *   dst[r] = RoPE(src[idx[r]], positions[idx[r]])   (a zero row where idx[r] < 0)
 * Source: guijiagi.com tag page "Ring Attention", article on the evolution of
 * long-context techniques, section 1.2 "RoPE": RoPE(x, m) = x e^{i m theta},
 * theta_i = base^(-2i/d) (i = 0 .. d/2-1), real form
 * x*cos + rotate_half(x)*sin, rotate_half(x1, x2) = (-x2, x1): component j and
 * component j + d/2 of each head are the real and imaginary parts of the j-th
 * complex number, turned by the angle m * theta_j.
 *
 * src        device [src_rows, H, d] of dt (RA_BF16 or RA_F32), 16-byte aligned.
 * idx        device int32 [rows] (e.g. the perm of ra_zigzag_partition), or
 *            NULL for the identity (then rows == src_rows, and dst may be src
 *            itself: the rotation is done in place).
 * positions  device int32 [src_rows]: the position m of each SOURCE row (its
 *            index inside its own sequence), in [0, 2^24).
 * base       the RoPE base (10000 on the page), finite and > 1.
 * dst        device [rows, H, d] of dt out, 16-byte aligned; must not overlap
 *            src when idx is given.
 * d must be a multiple of 16 (bf16) or 8 (fp32), at most 256.  The rotation
 * is computed in fp32 (angles reduced to turns with an error-free product, so
 * their error does not grow with the position) and rounded once to dt.
 * An idx >= src_rows or a position outside [0, 2^24) is a device-side bounds
 * error (RA_ERR_DEVICE_BOUNDS recorded; the row is zero-filled, resp. the
 * position taken as 0).
 * ---------------------------------------------------------------------- */
ra_status ra_rope_gather(const void* src, int64_t src_rows, int32_t H, int32_t d, ra_dtype dt,
                         const int32_t* idx, int64_t rows, const int32_t* positions, double base,
                         void* dst, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_ring_attn_fwd -- causal or full GQA attention forward computed in ring
 * order over N virtual context-parallel ranks with blockwise online softmax.
 * Sources: "Parallelism-CP" diagram (Q/K/V split along the sequence, K/V
 * rotate on a ring, every Q block meets every K/V block); guijiagi.com
 * "Ring Attention" tag page (ring step t: rank i uses the K/V of rank
 * (i - t) mod N; blockwise decomposition with running max and running sum);
 * vLLM-Ascend "Context Parallel (CP)" head-tail partition (rank r owns chunks
 * r and 2N-1-r).  The result equals full softmax attention.
 *
 * q    device [B*S, Hq, d]  (dtype dt), token order per `layout`.
 * k, v device [B*S, Hkv, d] (dtype dt), same token order.
 * o    device [B*S, Hq, d]  out, dtype dt, same token order.
 * lse  device float [B*S, Hq] out: natural-log sum of exp(scaled scores).
 * Query head h reads K/V head h / (Hq/Hkv).  scale <= 0 means 1/sqrt(d).
 * causal != 0: the query at original position i sees keys j <= i.
 * Requirements: B, Hq, Hkv, S >= 1; Hq % Hkv == 0; S % (2*n_ranks) == 0;
 * B*S < 2^31; pointers 16-byte aligned.  d must be 64 or 128
 * (RA_ERR_UNSUPPORTED otherwise).  RA_BF16 runs on the tensor cores
 * (tcgen05, fp32 accumulation); RA_F32 runs an exact fp32 SIMT kernel.
 * ---------------------------------------------------------------------- */
ra_status ra_ring_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d,
                           ra_dtype dt, int32_t causal, int32_t n_ranks, float scale,
                           ra_layout layout, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_ring_attn_fwd_varlen -- ring-order attention over several requests of
 * different lengths in one call, on the layout the head-tail partition
 * gathers them to (ra_zigzag_partition + ra_gather_rows with the same
 * seq_lens and n_ranks).
 * Sources: as ra_ring_attn_fwd; vLLM-Ascend developer guide "Context
 * Parallel (CP)", PCP head-tail token partition (each request padded to a
 * multiple of 2*pcp, its parts paired first-with-last, the gathered buffer
 * rank-major over requests).
 *
 * seq_lens  host int64 [num_seqs] real lengths L_b >= 0 (1 <= num_seqs <= 256).
 *           Request b is padded to L'_b = ceil(L_b/2N)*2N and cut into chunks
 *           of c_b = L'_b/2N tokens.
 * q, k, v   device bf16 [G, Hq|Hkv, d], G = sum_b L'_b rows in gathered order:
 *           rank-major, then request, then chunk r and chunk 2N-1-r of it.
 * o, lse    device out, same row order ([G, Hq, d] bf16 and [G, Hq] fp32).
 *           Rows of padding positions get the attention of a query at that
 *           position (the restore index drops them).
 * Each request attends to its own keys only; keys at padding positions
 * (>= L_b) are masked; causal compares original positions.  Runs the
 * adjacent-tile tcgen05 kernel (any Hq/Hkv); reads the device's SM count.
 * Errors: as ra_ring_attn_fwd; RA_ERR_UNSUPPORTED for RA_F32 or d not in
 * {64, 128}; a total padded length >= 2^31 is RA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
ra_status ra_ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const int64_t* seq_lens, int32_t num_seqs, int32_t Hq, int32_t Hkv,
                                  int32_t d, ra_dtype dt, int32_t causal, int32_t n_ranks, float scale,
                                  ra_stream stream);

/* Same as ra_ring_attn_fwd with an explicit bf16 kernel variant:
 * 0 = automatic (2 when Hq/Hkv is even, else 3);
 * 1 = one query head per CTA (mirrored pair of query tiles, 128-key tiles,
 *     P via shared memory);
 * 2 = two query heads of one GQA group per CTA sharing every 128-key K/V tile
 *     (needs an even Hq/Hkv; P stays in tensor memory);
 * 3 = two adjacent 128-row query tiles of one head per CTA sharing every K/V
 *     tile (any Hq/Hkv; same pipeline as 2).  Each call on this variant reads
 *     the current device's SM count to size its grid.
 * The variant is ignored for RA_F32.  All variants agree to rounding. */
ra_status ra_ring_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d,
                              ra_dtype dt, int32_t causal, int32_t n_ranks, float scale,
                              ra_layout layout, int32_t variant, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_ring_schedule_counts -- the (query tile, key tile) classification the
 * bf16 ring kernel uses, counted per virtual rank on the device by the same
 * schedule code: counts[r*3 + {0,1,2}] = tile pairs processed without mask,
 * with the causal diagonal mask, and skipped.  Tiles are 128 tokens, cut per
 * chunk (the last tile of a chunk may be shorter).
 * counts  device int64 [n_ranks*3] out.  Same size rules as ra_ring_attn_fwd.
 * ---------------------------------------------------------------------- */
ra_status ra_ring_schedule_counts(int32_t S, int32_t n_ranks, int32_t causal, int64_t* counts,
                                  ra_stream stream);

/* Same with an explicit key-tile length (64 or 128; the attention kernels use
 * 128).  Query tiles are always 128 rows. */
ra_status ra_ring_schedule_counts_ex(int32_t S, int32_t n_ranks, int32_t causal, int32_t kv_tile,
                                     int64_t* counts, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_attn_block_fwd -- partial attention of one query block against one key
 * block: the computation of one ring step (a rank's Q against the K/V block it
 * holds) or of one segment of a chunked prefill, whose partials ra_lse_merge
 * combines.  Sources: guijiagi.com "Ring Attention" tag page (per-step partial
 * attention, blockwise decomposition); vLLM-Ascend "Context Parallel (CP)",
 * chunked prefill (segments of bounded KV, online-softmax update per segment).
 *
 * q        device bf16 [Tq, Hq, d]: queries at positions q_pos0 .. q_pos0+Tq-1.
 * k, v     device bf16 [Tk, Hkv, d]: keys at positions k_pos0 .. k_pos0+Tk-1.
 * o_part   device float [Tq, Hq, d] out: softmax-weighted V over the visible keys
 *          of this block (normalised by the block's own sum), 0 if none.
 * lse_part device float [Tq, Hq] out: natural-log sum of exp(scaled scores)
 *          over the visible keys, -inf if none.
 * causal != 0: key position j is visible to query position i iff j <= i.
 * Same GQA mapping, scale and d rules as ra_ring_attn_fwd; bf16 only.
 * ---------------------------------------------------------------------- */
ra_status ra_attn_block_fwd(const void* q, const void* k, const void* v, int32_t Tq, int32_t Tk,
                            int32_t Hq, int32_t Hkv, int32_t d, int64_t q_pos0, int64_t k_pos0,
                            int32_t causal, float scale, float* o_part, float* lse_part,
                            ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_ring_step_fwd -- one step of a ring across devices, on the rank that runs
 * it: its queries against the K/V block it holds at this step, folded into its
 * running result.  Sources: "Parallelism-CP" diagram (each card computes its
 * own Q against the K/V blocks that rotate around the ring); guijiagi.com
 * "Ring Attention" tag page (ring topology: at step t rank i holds the block
 * of rank (i - t) mod N; blockwise decomposition, a partial over some keys is
 * carried by its log-sum-exp); vLLM-Ascend "Context Parallel (CP)" head-tail
 * partition (rank r holds chunks r and 2N-1-r).
 *
 * Local layout (what the head-tail partition gives a rank): per sequence
 * (B of them), the rank's first chunk then its second, c rows each; the row of
 * (sequence b, half h, offset o) is (b*2 + h)*c + o.
 * q          device bf16 [B*2c, Hq, d]: rank `rank`'s queries (chunks rank and
 *            2N-1-rank of each sequence).
 * k, v       device bf16 [B*2c, Hkv, d]: the block held, i.e. rank `src`'s
 *            local K/V (chunks src and 2N-1-src).
 * o_in, lse_in  device fp32 [B*2c, Hq, d] and [B*2c, Hq]: the running result
 *            (normalised O and its LSE) of the steps so far, or both NULL at
 *            the rank's first step.
 * o_out      device [B*2c, Hq, d] out in out_dt; lse_out device fp32
 *            [B*2c, Hq] out.  o_out may be o_in when out_dt is RA_F32 and
 *            lse_out may be lse_in (the running result updated in place); a
 *            bf16 o_out is the final output, given at the last step.
 * Result: the merge of the running result with this block's partial,
 * LSE = ln(e^{LSE_in} + e^{LSE_p}), O = e^{LSE_in - LSE} O_in + e^{LSE_p - LSE} O_p,
 * where (O_p, LSE_p) is attention over the keys of the block visible to each
 * query (causal != 0: original key position <= query position).  Rows that
 * see no key of the block keep the running result (O 0, LSE -inf without one).
 * Over the N steps (src = (rank - t) mod N, or any order) the result is the
 * rank's rows of full attention.  Query head h reads K/V head h / (Hq/Hkv);
 * scale <= 0 means 1/sqrt(d).  Even Hq/Hkv runs two heads per CTA, odd runs two
 * adjacent query tiles of one head per CTA.
 * Errors: B, Hq, Hkv, c < 1; Hq % Hkv != 0; rank or src outside [0, n_ranks);
 * o_in without lse_in or the reverse; a bf16 o_out equal to o_in; pointers
 * not 16-byte aligned (lse 4-byte); B*2c >= 2^31 -> RA_ERR_INVALID_ARG;
 * d not in {64, 128} -> RA_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
ra_status ra_ring_step_fwd(const void* q, const void* k, const void* v, int32_t B, int32_t Hq,
                           int32_t Hkv, int32_t c, int32_t d, int32_t n_ranks, int32_t rank,
                           int32_t src, int32_t causal, float scale, const float* o_in,
                           const float* lse_in, void* o_out, ra_dtype out_dt, float* lse_out,
                           ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_segmented_prefill_fwd -- chunked prefill with a bounded KV segment per
 * round (vLLM-Ascend "Context Parallel (CP)", chunked prefill, segmented
 * AllGatherKV): the key range [0, Tk) is cut into segments of seg_tokens; each
 * segment gives partials (ra_attn_block_fwd) and the partials are merged
 * (ra_lse_merge).  The result equals attention of the query block over all
 * Tk keys.
 *
 * q [Tq, Hq, d] at positions q_pos0..; k, v [Tk, Hkv, d] at positions 0..Tk-1
 * (bf16, device).  o [Tq, Hq, d] out in out_dt; lse [Tq, Hq] fp32 out (may be
 * NULL).  workspace: ra_segmented_prefill_workspace_size() bytes, 16-byte
 * aligned (the per-segment fp32 partials).
 * ---------------------------------------------------------------------- */
ra_status ra_segmented_prefill_workspace_size(int32_t Tq, int32_t Tk, int32_t Hq, int32_t d,
                                              int32_t seg_tokens, size_t* bytes);

ra_status ra_segmented_prefill_fwd(const void* q, const void* k, const void* v, int32_t Tq,
                                   int32_t Tk, int32_t Hq, int32_t Hkv, int32_t d, int64_t q_pos0,
                                   int32_t causal, float scale, int32_t seg_tokens, void* o,
                                   ra_dtype out_dt, float* lse, void* workspace, size_t ws_bytes,
                                   ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_lse_merge -- merge P partial attention results (the update of a
 * cp_lse_ag_out_rs-style gather: vLLM-Ascend "Context Parallel (CP)", DCP
 * decode; weights from the blockwise decomposition of the "Ring Attention"
 * tag page):  LSE = ln sum_p e^{LSE_p},  O = sum_p e^{LSE_p - LSE} O_p.
 * A partial with LSE_p = -inf has weight 0 and its O_p is not read; if every
 * partial is -inf the result is O = 0, LSE = -inf.
 *
 * o_parts   device float [P, T, H, d]; lse_parts device float [P, T, H].
 * o_out     device [T, H, d] out in out_dt; lse_out device float [T, H] out
 *           (may be NULL).  Requires P >= 1, d % 4 == 0, 16-byte aligned.
 * ---------------------------------------------------------------------- */
ra_status ra_lse_merge(const float* o_parts, const float* lse_parts, int32_t P, int64_t T,
                       int32_t H, int32_t d, void* o_out, ra_dtype out_dt, float* lse_out,
                       ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_slot_mapping -- interleaved context-parallel KV-cache slot mapping.
 * Source: vLLM-Ascend "Context Parallel (CP)", section "Block table":
 * V = block_size*pcp*dcp; for token position x: vb = x / V, o = x % V,
 * lbi = o / interleave, device = lbi % (pcp*dcp),
 * offset = (lbi / (pcp*dcp))*interleave + o % interleave,
 * slot = block_table[request][vb]*block_size + offset on that device.
 *
 * query_start_loc device int32 [R+1]: tokens of request q are
 *                 [query_start_loc[q], query_start_loc[q+1]) (non-decreasing,
 *                 query_start_loc[0] = 0, query_start_loc[R] = T).
 * positions       device int32 [T]: position x of each token in its request.
 * block_table     device int32 [R, max_vblocks]: physical block id of each
 *                 virtual block (the same id is used in every device's pool).
 * slot_out        device int32 [pcp*dcp, T] out: slot on each device, -1 where
 *                 the device does not store the token.
 * Errors: block_size % interleave != 0 -> RA_ERR_INVALID_ARG (the page's
 * rule); a token whose virtual block is >= max_vblocks or whose block id is
 * negative -> RA_ERR_DEVICE_BOUNDS (slot -1 everywhere).
 * ---------------------------------------------------------------------- */
ra_status ra_cp_slot_mapping(const int32_t* query_start_loc, const int32_t* positions,
                             const int32_t* block_table, int32_t max_vblocks, int32_t R,
                             int64_t T, int32_t block_size, int32_t interleave, int32_t pcp,
                             int32_t dcp, int32_t* slot_out, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_kv_scatter -- write token K/V rows into the sharded paged cache at the
 * slots of ra_cp_slot_mapping (the cache write that slot_mapping drives).
 *
 * k, v      device [T, Hkv, d] (dtype dt).
 * slot      device int32 [W, T] from ra_cp_slot_mapping (W = pcp*dcp).
 * k_cache, v_cache device [W, num_blocks, Hkv, block_size, d] (dtype dt):
 *           device w, block b, head g, in-block slot s is one d-vector.
 * A slot outside [0, num_blocks*block_size) is a device bounds error.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_kv_scatter(const void* k, const void* v, const int32_t* slot, void* k_cache,
                           void* v_cache, int64_t T, int32_t W, int32_t Hkv, int32_t d,
                           int32_t block_size, int64_t num_blocks, ra_dtype dt, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_kv_gather -- read token rows back out of the sharded paged cache in
 * any order: the reorg that makes each request's KV contiguous after the
 * context all-gather (vLLM-Ascend "Context Parallel (CP)", DCP chunked
 * prefill, MLA backend: all_gather of the context KV, then reorg_kvcache).
 * Row t of the outputs is token positions[t] of its request (query_start_loc
 * as in ra_cp_slot_mapping), located with the block-table formula.
 *
 * k_cache, v_cache device [W, num_blocks, Hkv, block_size, d] (dtype dt).
 * k_out, v_out     device [T, Hkv, d] out.
 * A virtual block >= max_vblocks or a block id outside [0, num_blocks) is a
 * device bounds error (the row is zero-filled).  block_size % interleave != 0
 * -> RA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_kv_gather(const void* k_cache, const void* v_cache, const int32_t* block_table,
                          int32_t max_vblocks, const int32_t* query_start_loc,
                          const int32_t* positions, int32_t R, int64_t T, int32_t Hkv, int32_t d,
                          int32_t block_size, int32_t interleave, int32_t pcp, int32_t dcp,
                          int64_t num_blocks, ra_dtype dt, void* k_out, void* v_out,
                          ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_decode -- one-token decode over the sharded paged cache: split-KV
 * partials per (request, device, split) followed by ra_lse_merge.
 * Source: vLLM-Ascend "Context Parallel (CP)", DCP decode and PCP decode
 * (attention over the local KV shard, then cp_lse_ag_out_rs); on one GPU all
 * W = pcp*dcp devices are virtual and every partial is merged at once.
 *
 * q           device bf16 [R, Hq, d] (the query token of each request).
 * k_cache, v_cache device bf16 [W, num_blocks, Hkv, block_size, d].
 * block_table device int32 [R, max_vblocks]; ctx_lens device int32 [R]: the
 *             query of request r attends its tokens 0..ctx_lens[r]-1.
 * split_blocks virtual blocks per split (>= 1): partial p = w*n_splits + s
 *             covers device w's blocks of virtual blocks
 *             [s*split_blocks, (s+1)*split_blocks), n_splits =
 *             ceil(max_vblocks/split_blocks).
 * o           device [R, Hq, d] out (out_dt); lse device float [R, Hq] out
 *             (may be NULL).
 * workspace   device scratch of ra_cp_decode_workspace_size() bytes
 *             (16-byte aligned): the fp32 partials.
 * Requires d in {64,128}, Hq % Hkv == 0, Hq/Hkv <= 8,
 * block_size % interleave == 0, every ctx_lens[r] <= max_vblocks*V.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_decode_workspace_size(int32_t R, int32_t Hq, int32_t d, int32_t max_vblocks,
                                      int32_t pcp, int32_t dcp, int32_t split_blocks,
                                      size_t* bytes);

ra_status ra_cp_decode(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                       int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                       int32_t interleave, int32_t pcp, int32_t dcp, int32_t max_vblocks,
                       int64_t num_blocks, float scale, int32_t split_blocks, void* o,
                       ra_dtype out_dt, float* lse, void* workspace, size_t ws_bytes,
                       ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_decode_partials -- the split-KV partials of the devices whose cache
 * shards the caller holds, unmerged: what one device computes before the
 * cp_lse_ag_out_rs merge across devices.  Source: vLLM-Ascend "Context
 * Parallel (CP)", DCP decode (each device attends over its local KV shard and
 * returns its output with its LSE) and section "Block table" (which device
 * stores which token).
 *
 * q, block_table, ctx_lens, sizes, scale, split_blocks: as ra_cp_decode.
 * dev0, n_dev  the cache holds devices dev0 .. dev0+n_dev-1 of W = pcp*dcp
 *             (all of them: dev0 = 0, n_dev = W; one device w: dev0 = w,
 *             n_dev = 1).
 * k_cache, v_cache device bf16 [n_dev, num_blocks, Hkv, block_size, d]:
 *             their shards, in that order.
 * o_parts     device float [P, R, Hq, d] out, lse_parts device float [P, R, Hq]
 *             out, P = n_dev * n_splits: partial p = (w - dev0)*n_splits + s
 *             covers device w's tokens of virtual blocks [s*split_blocks,
 *             (s+1)*split_blocks), O normalised by its own sum.  A partial
 *             with no token has LSE -inf and its O is not written.
 * n_parts_out host int32 out (may be NULL): P.  With o_parts and lse_parts
 *             both NULL only P is returned and nothing is launched (the
 *             other arguments are checked as for a launch).
 * Errors: as ra_cp_decode; [dev0, dev0+n_dev) outside [0, W) is
 * RA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                                int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                                int32_t interleave, int32_t pcp, int32_t dcp, int32_t dev0,
                                int32_t n_dev, int32_t max_vblocks, int64_t num_blocks, float scale,
                                int32_t split_blocks, float* o_parts, float* lse_parts,
                                int32_t* n_parts_out, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_lse_rescale -- step 2 of cp_lse_ag_out_rs on device w of W: after the
 * all-gather of every device's LSE, scale this device's output by its merge
 * weight and lay it out for the reduce-scatter over heads.  Source:
 * vLLM-Ascend "Context Parallel (CP)", DCP decode (cp_lse_ag_out_rs:
 * all-gather of the LSEs, local update of the output, reduce-scatter); the
 * weights e^{LSE_w - LSE} of the blockwise decomposition ("Ring Attention" tag
 * page).  Steps 1 and 3 are collectives of the caller's communication library.
 *
 * o_local   device float [R, Hq, d]: device w's output over its own keys
 *           (normalised; e.g. ra_lse_merge of its ra_cp_decode_partials).
 * lse_all   device float [W, R, Hq]: every device's LSE, device w's at w.
 * o_scaled  device float [W, R, Hq/W, d] out: slot v holds heads
 *           [v*Hq/W, (v+1)*Hq/W) of e^{LSE_w - LSE} O_w, LSE = ln sum_v e^{LSE_v}
 *           (0 where LSE_w or LSE is -inf; o_local is not read there).  Summed
 *           over devices, slot v is device v's merged output.
 * lse_total device float [R, Hq/W] out (may be NULL): LSE of this device's
 *           heads [w*Hq/W, (w+1)*Hq/W).
 * Requires 0 <= w < W, Hq % W == 0, d % 4 == 0 (RA_ERR_UNSUPPORTED otherwise),
 * o_local and o_scaled 16-byte aligned.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_lse_rescale(const float* o_local, const float* lse_all, int32_t W, int32_t w, int64_t R,
                            int32_t Hq, int32_t d, float* o_scaled, float* lse_total, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_head_split -- the all-to-all form of the decode merge across W
 * devices: device w lays out its output and LSE by the device that keeps each
 * head, so that one all-to-all of o_split and lse_split hands every device the
 * W partials of its own heads, which ra_lse_merge (P = W) then merges.
 * Source: vLLM-Ascend "Context Parallel (CP)", DCP decode and PCP decode (the
 * partial outputs and LSEs are exchanged by an all-to-all as an alternative to
 * cp_lse_ag_out_rs).
 *
 * o_local   device float [R, Hq, d]: this device's output over its own keys.
 * lse_local device float [R, Hq]: its LSE (-inf: no key; O is not read).
 * o_split   device float [W, R, Hq/W, d] out: slot v holds heads
 *           [v*Hq/W, (v+1)*Hq/W) of o_local (0 where the LSE is -inf).
 * lse_split device float [W, R, Hq/W] out: the same heads' LSEs.
 * Requires Hq % W == 0, d % 4 == 0 (RA_ERR_UNSUPPORTED otherwise), o_local and
 * o_split 16-byte aligned.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_head_split(const float* o_local, const float* lse_local, int32_t W, int64_t R, int32_t Hq,
                           int32_t d, float* o_split, float* lse_split, ra_stream stream);

/* ------------------------------------------------------------------------
 * ra_cp_decode_noalloc -- ra_cp_decode for callers that cannot allocate
 * device memory on the decode path (a runtime that reserves all device memory
 * at start-up and forbids allocation afterwards, an allocator that cannot
 * hand out raw scratch, a process whose device footprint must stay fixed).
 * The pages have no counterpart of this entry point; it only changes where
 * the scratch lives.
 *
 * Same arguments and results as ra_cp_decode, without workspace/ws_bytes:
 * the fp32 partials go to a fixed 32 MiB scratch array inside the library's
 * device memory, which every GPU that loads the library holds until exit.
 * No call allocates device memory through cudaMalloc, cudaFree or an
 * allocating library routine.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it for that
 *   device's context (a context created again after a reset is looked up
 *   again).  Under lazy module loading, CUDA's default, that first call also
 *   loads the decode module and so commits the array's 32 MiB; a caller that
 *   may not allocate after start-up makes one warm-up call per device at
 *   start-up, or runs with CUDA_MODULE_LOADING=EAGER.  Calls after the first
 *   commit nothing.  Make the first call before any stream capture.
 * - A decode whose partials need more than 32 MiB
 *   (ra_cp_decode_workspace_size) is rejected with RA_ERR_INVALID_ARG; a
 *   larger split_blocks makes it smaller.
 * - All calls share the array and it keeps the last call's contents.  Nothing
 *   in it needs to start at zero (every partial's LSE is written before it is
 *   read, and a partial's O is read only if the same call wrote it).  Calls
 *   whose work overlaps on the GPU (e.g. on two streams) race on the array.
 * ---------------------------------------------------------------------- */
ra_status ra_cp_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                               int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                               int32_t interleave, int32_t pcp, int32_t dcp, int32_t max_vblocks,
                               int64_t num_blocks, float scale, int32_t split_blocks, void* o,
                               ra_dtype out_dt, float* lse, ra_stream stream);

/* ------------------------------------------------------------------------
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nobody arrives at, for at most `limit_cycles` SM clock cycles,
 * then records RA_ERR_TIMEOUT in the device error word and returns.  The
 * context stays usable.  Used by the tests to check failure detection.
 * ---------------------------------------------------------------------- */
ra_status ra_selftest_wait_timeout(int64_t limit_cycles, ra_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
