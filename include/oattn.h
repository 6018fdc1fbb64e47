/*
 * oattn.h - C ABI of the online-softmax attention library for NVIDIA GB300 (sm_103a).
 *
 * Three operations (each also with an optional Boolean mask), all asynchronous on the
 * caller's CUDA stream:
 *
 *   attn_fwd         single-pass tiled scaled-dot-product attention forward with the
 *                    online-softmax recurrence ("A3. Tiled attention with online
 *                    normalization", sections "Keep three quantities for each query row"
 *                    and "Masks that preserve the recurrence"; "Streaming attention and
 *                    online state", section "Online statistics").
 *   attn_fwd_splitk  the same attention with the key axis cut into P partitions; each
 *                    partition writes its locally normalised output O_p and a base-2
 *                    log-sum-exp lse_p ("fa4_splitk_combine", workspace layout), then,
 *                    when an output pointer is given, the partitions are merged.
 *   splitk_combine   the LSE-weighted merge of P partitions ("fa4_splitk_combine",
 *                    the per row-head formulas for m*, global_lse, scale_p and O[d]).
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, o, lse, o_partial, lse_partial are DEVICE pointers owned by
 *     the caller; the library never allocates, frees or retains them.  Every tensor is
 *     dense and row-major (last index contiguous).  16-bit and float32 tensors must start
 *     on a 16-byte boundary; float LSE arrays on a 4-byte boundary.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is enqueued
 *     and the call returns without synchronising.  The attention kernels are launched
 *     as programmatic dependents of the previous kernel on the stream: they may be
 *     scheduled while it finishes and wait for its completion before touching memory.
 *     attn_fwd (key tiles of 128) and attn_fwd_masked_blocks launch one CTA per SM,
 *     each walking a share of the (head, query-tile pair) work; attn_fwd_masked, the
 *     split-K and the 32/64-key forms launch one CTA per query-tile pair.  Argument errors are returned before anything is
 *     launched; a failed launch returns OATTN_ERR_CUDA.
 *   - Scores are s = scale * q.k.  Causal masking keeps key index <= query index (the
 *     diagonal included) and requires equal query and key lengths.
 *   - A query row with no visible key produces output +0 and LSE -inf.
 *   - Arithmetic: FP32 running max, sum and numerator; exp as ex2.approx of a scaled
 *     argument; the probabilities are rounded to the input dtype (round to nearest
 *     even) before the P.V product while the denominator sums the unrounded FP32 values.
 *   - Every wait inside the kernels is bounded.  A wait that gives up records a code in
 *     a device status word and the kernel returns early (its outputs are then
 *     undefined); read and clear that word with oattn_device_error().
 *   - Calls from several host threads are safe: the one-time set-up on each device
 *     (the status word's address, kernel attributes, the host entry point's streams) is
 *     guarded.  Calls that share a buffer or a workspace are not ordered by the library.
 */
#ifndef OATTN_H
#define OATTN_H

/* The library is built with hidden symbol visibility; these entry points alone are
 * exported. */
#if defined(__GNUC__)
#define OATTN_API __attribute__((visibility("default")))
#else
#define OATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*` */

typedef enum {
  OATTN_OK = 0,
  OATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad dtype     */
  OATTN_ERR_UNSUPPORTED = 2, /* valid request outside the compiled instances (e.g. D=96) */
  OATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a kernel launch failed     */
  OATTN_ERR_TIMEOUT = 4      /* reported by oattn_device_error(): a bounded wait gave up */
} oattn_status;

typedef enum { OATTN_F16 = 0, OATTN_BF16 = 1, OATTN_F32 = 2 } oattn_dtype;

/*
 * attn_fwd - O = softmax(scale * Q K^T [causal mask]) V and the per-row log-sum-exp.
 *
 *   q, k, v  [B, H, N, D] dtype (f16 or bf16); o [B, H, N, D] same dtype.
 *   lse      [B, H, N] float32, natural-log log-sum-exp of the scaled scores of each row
 *            (M + ln L); may be NULL.
 *   D in {16, 32, 64, 128}; N >= 0 (N == 0 is a no-op); B, H >= 1; scale finite, > 0.
 * Returns OATTN_OK, OATTN_ERR_INVALID_ARG or OATTN_ERR_UNSUPPORTED (dtype f32, other D),
 * or OATTN_ERR_CUDA.
 */
OATTN_API oattn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int D, int causal, float scale,
                                oattn_dtype dtype, struct CUstream_st* stream);

/*
 * attn_fwd_host - attn_fwd with the inputs and outputs in HOST memory: the heads are cut
 * into chunks, and each chunk's copy in (host -> device), attention and copy out
 * (device -> host) run on three internal streams so that one chunk's copies overlap its
 * neighbours' attention.  Same result as attn_fwd, bit for bit.
 *
 *   q_h, k_h, v_h  [B, H, N, D] host inputs (pinned memory, or the copies do not overlap).
 *   o_h            [B, H, N, D] host output;  lse_h  [B, H, N] float32 host output or NULL.
 *   q_d, k_d, v_d, o_d, lse_d  device staging buffers of the same shapes, owned by the
 *                  caller (lse_d NULL exactly when lse_h is NULL).
 *   chunk_heads    heads (of the flattened B*H) per chunk; 0 picks ceil(B*H/8).
 * The work starts after everything already queued on `stream`, and work queued on `stream`
 * afterwards waits for the last copy out.  The first call on a device creates three
 * streams and four events there (kept until the process exits).  Calls on one device
 * share them: a call holds a per-device lock while it enqueues, so calls from several host
 * threads are safe and their work runs one after the other on the internal streams (each
 * still ordered after its own `stream`).  The staging buffers of calls that may overlap
 * must not alias.  Errors as attn_fwd.
 */
OATTN_API oattn_status attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                                     float* lse_h, void* q_d, void* k_d, void* v_d, void* o_d,
                                     float* lse_d, int B, int H, int N, int D, int causal, float scale,
                                     oattn_dtype dtype, int chunk_heads, struct CUstream_st* stream);

/*
 * attn_fwd_bn - attn_fwd with an explicit key-tile width block_n in {32, 64, 128}
 * ("A3. Tiled attention ...", section "Implement in four stages": BN is exposed as a
 * tuning choice).  block_n == 0 picks the default (128).  Results differ from attn_fwd
 * only by floating-point summation order.
 */
OATTN_API oattn_status attn_fwd_bn(const void* q, const void* k, const void* v, void* o, float* lse,
                                   int B, int H, int N, int D, int causal, float scale,
                                   oattn_dtype dtype, int block_n, struct CUstream_st* stream);

/*
 * attn_fwd_splitk - attention with the key axis split into P partitions.
 *
 *   q [B, H, Nq, D]; k, v [B, H, Nkv, D]; dtype f16 or bf16; D in {16, 32, 64, 128}.
 *   Partition p holds keys [p*C, min((p+1)*C, Nkv)) with
 *   C = splitk_chunk(Nkv, P) = ceil(ceil(Nkv/P)/128)*128; trailing partitions may be empty.
 *   o_partial [P, B*H*Nq, D] of partial_dtype (f32, or the input dtype): partition p's
 *            output normalised by its own sum; row-heads are flattened in (b, h, n)
 *            order, which for Nq == 1 is the (token, head) order of the combine page.
 *   lse_partial [P, B*H*Nq] float32, base-2: lse_p = m_p + log2(l_p) with m_p the
 *            partition's row max of scale*q.k*log2(e).  A (row, partition) with no
 *            visible key stores O_p = +0 and lse_p = -inf.
 *   o        NULL: stop after the partials.  Otherwise [B, H, Nq, D] dtype receives the
 *            merged attention output (splitk_combine over the partials).
 *   lse      NULL, or [B, H, Nq] float32 natural-log LSE of the merged result (needs o).
 *   1 <= P <= 256; causal requires Nq == Nkv.
 * o_partial and lse_partial are scratch owned by the caller and must not overlap q, k, v,
 * o or lse.
 */
OATTN_API oattn_status attn_fwd_splitk(const void* q, const void* k, const void* v, void* o, float* lse,
                                       int B, int H, int Nq, int Nkv, int D, int causal, float scale,
                                       oattn_dtype dtype, int P, void* o_partial, float* lse_partial,
                                       oattn_dtype partial_dtype, struct CUstream_st* stream);

/*
 * splitk_combine - merge P partitions by their base-2 LSEs ("fa4_splitk_combine").
 *
 *   o_partial   [P, rows*heads, depth] of in_dtype (f32, f16 or bf16), each partition
 *               normalised by its own sum; row-head index rh = row*heads + head.
 *   lse_partial [P, rows*heads] float32, base 2; -inf marks an empty partition.
 *   o           [rows*heads, depth] of out_dtype (f32, f16 or bf16).
 *   lse_out     NULL, or [rows*heads] float32 receiving global_lse (base 2).
 *   Per row-head: m* = max_p lse_p; global_lse = log2(sum_p 2^(lse_p - m*)) + m*;
 *   O[d] = sum_p 2^(lse_p - global_lse) * o_partial[p, rh, d].  Partitions whose lse_p is
 *   -inf contribute nothing; a row-head whose every lse_p is -inf gets O = +0 and
 *   global_lse = -inf.  o_partial must be finite where lse_p is finite.
 *   1 <= P <= 256; rows, heads >= 1; depth a power of two with depth*sizeof(in_dtype)
 *   between 32 and 1024 bytes (f32: 8..256, f16/bf16: 16..512).
 */
OATTN_API oattn_status splitk_combine(const void* o_partial, const float* lse_partial, void* o,
                                      float* lse_out, int P, int rows, int heads, int depth,
                                      oattn_dtype in_dtype, oattn_dtype out_dtype,
                                      struct CUstream_st* stream);

/*
 * attn_fwd_splitk_noalloc - attn_fwd_splitk for callers that cannot allocate device
 * memory (for example a plugin whose host framework owns all device memory through its
 * own pool, or a latency-critical caller that cannot afford the device synchronisation
 * an allocation may cause).  The reference pages have no counterpart for this entry
 * point; it only changes where the partition workspace lives.
 *
 *   Arguments as attn_fwd_splitk, without o_partial / lse_partial / partial_dtype: the
 *   float32 partials go to a fixed workspace inside the library (a device array of
 *   10 Mi + 256 Ki floats, 41 MiB, held on every GPU that loads the library until the
 *   process exits).  o is required when Nq > 0; lse may be NULL.
 *   Requires P * B*H*Nq * D <= 10485760 and P * B*H*Nq <= 262144, else returns
 *   OATTN_ERR_UNSUPPORTED before touching the device.  Every other argument is checked
 *   as attn_fwd_splitk checks it, empty problems (Nq == 0) included, with the same
 *   errors.
 *   The first call on a device looks up the workspace's device address (a host-side
 *   runtime call); make that first call before any stream capture.
 *   Every call uses the same workspace: calls that may overlap on the GPU (different
 *   streams, or different host threads on one device) race and must be serialised by
 *   the caller.  Each call rewrites every partial it reads, so no clearing is needed.
 */
OATTN_API oattn_status attn_fwd_splitk_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                               int B, int H, int Nq, int Nkv, int D, int causal, float scale,
                                               oattn_dtype dtype, int P, struct CUstream_st* stream);

/*
 * The optional Boolean M x N mask ("Streaming attention and online state", section
 * "Attention as a consumer": the worked attention kernel takes an optional Boolean input
 * mask of queries by keys).  The kernels read it packed, one bit per key:
 *
 *   a packed row holds attn_mask_words(Nkv) = 4*ceil(Nkv/128) 32-bit words; bit j of
 *   word w (value 1u << j) stands for key 32*w + j and is set when the key is visible.
 *   Bits at or past Nkv are ignored.  The mask is combined with the causal rule and
 *   the sequence bounds: a key is used when all three allow it.  A row whose every key
 *   is hidden gets output +0 and LSE -inf (the fully masked convention of "Streaming
 *   attention and online state", section "Online statistics").
 *
 *   In the masked entry points, row (b, h, q) of the mask starts at
 *   mask_bits + b*mask_stride_b + h*mask_stride_h + q*mask_stride_q (strides in 32-bit
 *   words, >= 0, multiples of 4; a stride of 0 shares the rows along that axis, e.g. one
 *   [N, Nkv] mask for every head, or a key-padding mask [B, Nkv] with mask_stride_h =
 *   mask_stride_q = 0).  mask_bits is a device pointer on a 16-byte boundary, owned by
 *   the caller and only read.
 */
OATTN_API int attn_mask_words(int Nkv);

/*
 * attn_mask_pack - pack a byte mask into the bit layout above.
 *
 *   mask  device bytes; row r (0 <= r < rows) is mask[r*row_stride .. r*row_stride + Nkv),
 *         nonzero = visible (a bool tensor's storage).  row_stride >= Nkv, in bytes.
 *   bits  device words, [rows, attn_mask_words(Nkv)], 16-byte aligned; every word is
 *         written (bits past Nkv as zero).
 * rows == 0 or Nkv == 0 is a no-op.  Returns OATTN_ERR_INVALID_ARG for negative sizes,
 * null or misaligned pointers or row_stride < Nkv.
 */
OATTN_API oattn_status attn_mask_pack(const void* mask, unsigned int* bits, long long rows, int Nkv,
                                      long long row_stride, struct CUstream_st* stream);

/*
 * attn_fwd_masked - attn_fwd (key tiles of 128) with the optional Boolean mask added.
 *   Arguments as attn_fwd, plus the packed mask and its strides (above); the mask is
 *   required (non-NULL) when N > 0.  Causal and mask may be combined.  Key tiles that
 *   no row of a block of 256 query rows sees are skipped, so a sliding window or key
 *   padding costs only the tiles it touches (the mask is scanned once per block).
 */
OATTN_API oattn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                                       int B, int H, int N, int D, int causal, float scale,
                                       oattn_dtype dtype, const unsigned int* mask_bits,
                                       long long mask_stride_b, long long mask_stride_h,
                                       long long mask_stride_q, struct CUstream_st* stream);

/*
 * The block summary of a packed mask: one bit per (mask head, block of 256 query rows,
 * key tile of 128 keys), set when some row of the block sees some key of the tile.  A
 * mask head is (b, h) with b taken as 0 when mask_stride_b == 0 and h taken as 0 when
 * mask_stride_h == 0 (a shared mask has a shared summary).  The words of mask head
 * (b, h) and block p are blocks[((b*Hm + h)*ceil(Nq/256) + p)*wpb .. + wpb) with
 * Hm = (mask_stride_h ? H : 1) and wpb = ceil(ceil(Nkv/128)/32); bit j of word i stands
 * for key tile 32*i + j.  The summary depends only on the mask: it is made once per mask
 * (as the packing is) and serves every call that uses that mask.
 *
 * attn_mask_blocks_words - words of the summary: (mask_stride_b ? B : 1) *
 *   (mask_stride_h ? H : 1) * ceil(Nq/256) * wpb; 0 when any size is <= 0.
 */
OATTN_API long long attn_mask_blocks_words(int B, int H, int Nq, int Nkv, long long mask_stride_b,
                                           long long mask_stride_h);

/*
 * attn_mask_blocks - write the block summary of the packed mask (strides as in the
 *   masked entry points) into `blocks`, a device array of attn_mask_blocks_words(...)
 *   32-bit words on a 4-byte boundary, owned by the caller; every word is written.  Reads
 *   rows q < Nq of each mask head.  Nq == 0 or Nkv == 0 is a no-op.  Returns
 *   OATTN_ERR_INVALID_ARG for negative sizes, null or misaligned pointers and bad
 *   strides, OATTN_ERR_UNSUPPORTED above 2^31 - 1 summary words.
 */
OATTN_API oattn_status attn_mask_blocks(const unsigned int* mask_bits, long long mask_stride_b,
                                        long long mask_stride_h, long long mask_stride_q, int B, int H,
                                        int Nq, int Nkv, unsigned int* blocks, struct CUstream_st* stream);

/*
 * attn_fwd_masked_blocks - attn_fwd_masked with the block summary of the same mask
 *   (attn_mask_blocks with Nq = Nkv = N, the same pointer, strides, B and H, written
 *   after the mask's last change; a stale summary leaves out tiles it should not).
 *   One CTA per SM walks its blocks and visits, in each block, only the key tiles the
 *   summary marks, so no mask scan precedes the key loop.  When a CTA's share of the
 *   summary exceeds 256 words (2 * ceil(units / SMs) * wpb, units = B*H*ceil(N/512) for
 *   causal, B*H*ceil(N/256) otherwise) the call runs as attn_fwd_masked.  Results are
 *   those of attn_fwd_masked.  Errors as attn_fwd_masked; blocks must be non-NULL and
 *   4-byte aligned when N > 0.
 */
OATTN_API oattn_status attn_fwd_masked_blocks(const void* q, const void* k, const void* v, void* o, float* lse,
                                              int B, int H, int N, int D, int causal, float scale,
                                              oattn_dtype dtype, const unsigned int* mask_bits,
                                              long long mask_stride_b, long long mask_stride_h,
                                              long long mask_stride_q, const unsigned int* blocks,
                                              struct CUstream_st* stream);

/*
 * attn_fwd_splitk_masked - attn_fwd_splitk with the optional Boolean mask (above) over
 *   the Nq x Nkv scores of each head.  A (row, partition) whose keys are all hidden
 *   stores O_p = +0 and lse_p = -inf, like an empty partition.  Nq == 1 reads only
 *   row q = 0 of each (b, h), so mask_stride_q is not used there.
 */
OATTN_API oattn_status attn_fwd_splitk_masked(const void* q, const void* k, const void* v, void* o,
                                              float* lse, int B, int H, int Nq, int Nkv, int D,
                                              int causal, float scale, oattn_dtype dtype, int P,
                                              void* o_partial, float* lse_partial,
                                              oattn_dtype partial_dtype, const unsigned int* mask_bits,
                                              long long mask_stride_b, long long mask_stride_h,
                                              long long mask_stride_q, struct CUstream_st* stream);

/*
 * attn_fwd_splitk_fused - attn_fwd_splitk with the merge done inside the attention
 * kernel instead of a second launch.  "fa4_splitk_combine" describes its kernel as the
 * traditional, unfused (workspace) merge; here the CTA that finishes last among the P
 * partitions of a group merges them ("Streaming attention and online state", Online
 * statistics: independent summaries merge by rescaling to a common maximum).  Groups are
 * row-heads for Nq == 1, and (head, 256 query rows) otherwise.
 *
 *   Arguments as attn_fwd_splitk, with o required, plus:
 *   counters   device uint32 array of at least attn_splitk_counters(B, H, Nq) words
 *              (B*H*Nq is always enough), 4-byte aligned, all ZERO before the first
 *              call.  Each call counts the finished partitions of a group there and
 *              the last one resets the word to zero, so a completed call leaves the
 *              array zero for the next one.  After a call that reported an error
 *              (oattn_device_error), clear the array again.  Calls that may overlap on
 *              the GPU must use different counter arrays.
 *   mask_bits  NULL, or the packed optional Boolean mask with its strides (as in
 *              attn_fwd_splitk_masked).
 * o_partial / lse_partial still receive every partition (the last CTA reads them back,
 * normally from L2); they and the counters are owned by the caller.
 */
OATTN_API int attn_splitk_counters(int B, int H, int Nq);

OATTN_API oattn_status attn_fwd_splitk_fused(const void* q, const void* k, const void* v, void* o,
                                             float* lse, int B, int H, int Nq, int Nkv, int D,
                                             int causal, float scale, oattn_dtype dtype, int P,
                                             void* o_partial, float* lse_partial,
                                             oattn_dtype partial_dtype, unsigned int* counters,
                                             const unsigned int* mask_bits, long long mask_stride_b,
                                             long long mask_stride_h, long long mask_stride_q,
                                             struct CUstream_st* stream);

/* Key chunk per partition used by attn_fwd_splitk (host-only, no GPU needed). */
OATTN_API int splitk_chunk(int Nkv, int P);

/* Human-readable name of a status code (static string). */
OATTN_API const char* oattn_status_string(oattn_status s);

/*
 * oattn_device_error - read and clear the device status word of the current device.
 * Synchronises the current device.  *code receives 0 when no bounded wait gave up
 * since the last call, else a nonzero site code; returns OATTN_ERR_TIMEOUT in that case,
 * OATTN_OK otherwise, or OATTN_ERR_CUDA if the device could not be queried.
 */
OATTN_API oattn_status oattn_device_error(int* code);

/*
 * oattn_selftest_wait - exercises the bounded-wait failure path on the device without a
 * fault: one thread waits for an mbarrier phase that can never complete (two arrivals
 * expected, one made); after the library's wait limit (2 s) the wait gives up, records
 * the site code OATTN_SELFTEST_SITE in the device status word and raises its CTA's abort
 * flag; a second warp, waiting on a barrier nothing arrives on, leaves through that flag.
 * The kernel then returns and the context stays usable: oattn_device_error() reports
 * OATTN_ERR_TIMEOUT with code OATTN_SELFTEST_SITE.
 *   flags  optional device array of 2 ints (NULL allowed): 1 where a wait completed,
 *          0 where it gave up (both 0 after a correct run).
 * Returns OATTN_OK once the kernel is enqueued, OATTN_ERR_INVALID_ARG for a misaligned
 * flags pointer, OATTN_ERR_CUDA for a failed launch.
 */
#define OATTN_SELFTEST_SITE 0x1F0
OATTN_API oattn_status oattn_selftest_wait(int* flags, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif
#endif /* OATTN_H */
