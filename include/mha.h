/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention forward.
 *
 * Operation (per batch b, head h, query row i):
 *
 *     out[b,h,i,:] = sum_j softmax_j( scale * q[b,h,i,:] . k[b,h,j,:] ) v[b,h,j,:]
 *
 * the scaled dot-product attention of "Attention Is All You Need", as stated
 * on the pages
 *   trishampatil.com      "Scaled Dot-Product Attention: Step by Step" (the
 *                         four steps: QK^T, divide by sqrt(d_k), row softmax,
 *                         weighted sum of V) and "Multi-Head Attention" (h
 *                         heads, each its own attention of width d_k = d_v);
 *   trishampatil.com      "Why Masking Is Required" (illegal logits -> -inf);
 *   alexdo.xyz            "Decoder block" (causal: i sees j <= i;
 *                         cross-attention: T queries x S keys, not causal)
 *                         and "Two masks, not one" (padded slots -> -inf);
 *   aicassindra.com       "A faithful layer in code" (per-head layout
 *                         [B, h, T, d_k] after the head split) and "Pitfalls
 *                         when reproducing the paper" (mask keys, not queries;
 *                         a fully masked row has no defined output).
 *
 * Every call enqueues GPU work on `stream` and returns; nothing is allocated,
 * nothing is synchronised, no host memory is touched besides the arguments.
 * The library holds no per-call state and is safe to call from several
 * threads at once.
 */
#ifndef MHA_GB300_H
#define MHA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and out (all four share it). */
typedef enum {
  MHA_DTYPE_F32 = 0,  /* float32 in, float32 out; CUDA-core FFMA, no TF32      */
  MHA_DTYPE_BF16 = 1  /* bfloat16 in, bfloat16 out (round to nearest even);
                         tensor-core products, float32 accumulation and softmax */
} mha_dtype;

/* mask_kind is a bit set. */
enum {
  MHA_MASK_NONE = 0,
  /* key j is allowed for query i only if j <= i (decoder self-attention);
     requires Lq == Lk */
  MHA_MASK_CAUSAL = 1,
  /* key j is allowed only if j < key_lengths[b] (padded source slots) */
  MHA_MASK_KEY_PADDING = 2,
  /* query rows i >= key_lengths[b] are padding: written as +0.0; requires
     Lq == Lk (self-attention over one padded sequence) */
  MHA_MASK_QUERY_PADDING = 4,
  /* generation with a key/value cache (alexdo.xyz, "How predictions are
     generated"): the Lq queries are the last Lq positions len - Lq .. len - 1
     of a sequence whose len keys are cached (len = key_lengths[b] with
     KEY_PADDING, else Lk); query i sees keys j <= len - Lq + i.  Any Lq, Lk;
     not combined with CAUSAL or QUERY_PADDING.  Queries before the cache's
     first position (len < Lq) have no key and are written as +0.0. */
  MHA_MASK_CAUSAL_TAIL = 8
};
/* encoder self-attention over padded sentences: KEY_PADDING | QUERY_PADDING;
   cross-attention over a padded source: KEY_PADDING; decoder: CAUSAL;
   decoder step over a key/value cache: CAUSAL_TAIL | KEY_PADDING. */

/* Memory layout of q, k, v and out (mha_fwd_ex; all four share it). */
enum {
  /* [B, heads, L, d]: the per-head layout after the head split and transpose
     (aicassindra.com, "A faithful layer in code") */
  MHA_LAYOUT_BHSD = 0,
  /* [B, L, heads, d]: the projection output viewed as heads, before the
     transpose, so no transpose copy is needed on either side of the call */
  MHA_LAYOUT_BSHD = 1
};

typedef enum {
  MHA_OK = 0,
  MHA_ERR_INVALID_ARGUMENT = 1, /* rejected before any launch              */
  MHA_ERR_UNSUPPORTED = 2,      /* valid, but no kernel for this shape/type */
  MHA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed        */
  MHA_ERR_TIMEOUT = 4           /* a kernel gave up waiting (device status) */
} mha_status;

/*
 * mha_fwd -- attention forward, asynchronous on `stream`.
 *
 * q    [B, H, Lq, d_k]  device pointer, contiguous row-major, 16-byte aligned
 * k    [B, H, Lk, d_k]  device pointer, contiguous row-major, 16-byte aligned
 * v    [B, H, Lk, d_v]  device pointer, contiguous row-major, 16-byte aligned
 * out  [B, H, Lq, d_v]  device pointer, contiguous row-major, 16-byte aligned;
 *                       written in full; must not overlap q, k, v or key_lengths
 * B, H, Lq, Lk          >= 0; a product B*H*Lq of 0 is a no-op; Lk == 0 (no
 *                       keys at all) writes +0.0 everywhere
 * d_k, d_v              > 0.  BF16: d_k == d_v, one of 64 or 128.
 *                       F32: 1..128 each.  Others: MHA_ERR_UNSUPPORTED
 * mask_kind             MHA_MASK_* bit set (see above)
 * key_lengths           device pointer to int32[B], required when a padding bit
 *                       is set (else ignored, may be NULL).  Read on the
 *                       device; values are clamped to [0, Lk].
 * scale                 multiplies every logit; pass 1/sqrt(d_k) for the
 *                       paper's scaling.  Any finite value (0 gives the mean of
 *                       the allowed values).
 * dtype                 mha_dtype
 * stream                cudaStream_t, or NULL for the legacy default stream
 *
 * Rows with no allowed key (key_lengths[b] == 0) and query-padding rows are
 * written as +0.0.  Keys and values at masked positions never influence the
 * result, provided they hold finite numbers.
 *
 * Ownership: every buffer belongs to the caller and must stay valid until the
 * enqueued work has run.  Errors: validation failures return before anything
 * is enqueued; MHA_ERR_CUDA reports a failed launch or driver call (the
 * runtime's sticky error, if any, is left for the caller to read).  Faults and
 * device-side timeouts surface at the caller's next synchronisation and in
 * mha_debug_status().
 */
int mha_fwd(const void *q, const void *k, const void *v, void *out,
            int B, int H, int Lq, int Lk, int d_k, int d_v,
            int mask_kind, const int32_t *key_lengths,
            float scale, int dtype, void *stream);

/*
 * mha_fwd_ex -- mha_fwd with shared key/value heads and a choice of layout.
 *
 * Grouped-query and multi-query attention are multi-head attention whose key
 * and value heads are shared by groups of query heads, or collapsed into one
 * (zeroshotmind.com, "Many heads, many subspaces"; trishampatil.com,
 * "Limitations of the Original Design").  Query head h reads key/value head
 * h / (H / H_kv):
 *
 *     out[b,h,i,:] = sum_j softmax_j( scale * q[b,h,i,:] . k[b,g,j,:] ) v[b,g,j,:],
 *     g = h / (H / H_kv)
 *
 * H_kv                  key/value heads, > 0 and dividing H (H_kv == H is
 *                       plain multi-head attention, H_kv == 1 multi-query)
 * layout                MHA_LAYOUT_BHSD: q [B, H, Lq, d_k], k [B, H_kv, Lk, d_k],
 *                       v [B, H_kv, Lk, d_v], out [B, H, Lq, d_v];
 *                       MHA_LAYOUT_BSHD: q [B, Lq, H, d_k], k [B, Lk, H_kv, d_k],
 *                       v [B, Lk, H_kv, d_v], out [B, Lq, H, d_v]
 *
 * Every other argument, the ownership rules and the error behaviour are those
 * of mha_fwd; an H_kv that does not divide H, or another layout value, is
 * MHA_ERR_INVALID_ARGUMENT.  mha_fwd(...) equals mha_fwd_ex with H_kv = H and
 * MHA_LAYOUT_BHSD.  The kernel choice depends on H_kv only through the
 * number of query rows per key/value head, (H / H_kv) * Lq (mha_fwd_path_ex),
 * and not on the layout.
 */
int mha_fwd_ex(const void *q, const void *k, const void *v, void *out,
               int B, int H, int H_kv, int Lq, int Lk, int d_k, int d_v, int layout,
               int mask_kind, const int32_t *key_lengths,
               float scale, int dtype, void *stream);

/*
 * mha_fwd_lse -- mha_fwd_ex that also stores each query row's softmax
 * statistics for the backward pass:
 *
 *     lse[b,h,i] = log2( sum_j 2^(scale * log2(e) * q[b,h,i,:] . k[b,g,j,:]) ),
 *
 * over the allowed keys j (the logarithm, in base 2, of the denominator of
 * step 3 of trishampatil.com, "Scaled Dot-Product Attention: Step by Step";
 * multiply by ln 2 for the natural logarithm).  Rows stored as +0.0 (query
 * padding, no allowed key) get +inf.  Training keeps these statistics from
 * the forward pass so that the backward pass need not recompute the scores a
 * second time (mha_bwd_lse).
 *
 * lse                   device pointer to float[B, H, Lq] (that order, whatever
 *                       the layout), 4-byte aligned, caller-owned; written in
 *                       full; must not overlap any other argument.  NULL is
 *                       MHA_ERR_INVALID_ARGUMENT unless B*H*Lq == 0.
 *
 * Every other argument, the ownership rules and the errors are those of
 * mha_fwd_ex; `out` is the same as mha_fwd_ex's.
 */
int mha_fwd_lse(const void *q, const void *k, const void *v, void *out, float *lse,
                int B, int H, int H_kv, int Lq, int Lk, int d_k, int d_v, int layout,
                int mask_kind, const int32_t *key_lengths,
                float scale, int dtype, void *stream);

/*
 * mha_linear_fwd -- y = x W + b, asynchronous on `stream`.
 *
 * The learned projection of token vectors that surrounds the attention
 * (trishampatil.com, "Multi-Head Attention": Q · W_i^Q with W_i^Q of shape
 * d_model x d_k; aicassindra.com, "A faithful layer in code": every linear
 * layer carries a bias).  Tensor-core products, fp32 accumulation, bf16 out.
 *
 * x    [M, K]  device pointer, row-major bf16, 16-byte aligned
 * w    [K, N]  device pointer, row-major bf16 (input-major), 16-byte aligned
 * b    [N]     device pointer, bf16, or NULL for no bias
 * y    [M, N]  device pointer, row-major bf16, 16-byte aligned; written in full;
 *              must not overlap x, w or b
 * M >= 0 (0 is a no-op); K, N > 0 and multiples of 8 (16-byte rows), else
 * MHA_ERR_UNSUPPORTED; dtype must be MHA_DTYPE_BF16 (F32: MHA_ERR_UNSUPPORTED).
 * Ownership and errors as for mha_fwd.
 */
int mha_linear_fwd(const void *x, const void *w, const void *b, void *y,
                   int M, int K, int N, int dtype, void *stream);

/* Bytes of device workspace mha_sublayer_fwd needs for these shapes (the
   projected q, k, v and the concatenated heads, bf16, each 256-byte aligned);
   0 for negative arguments. */
size_t mha_sublayer_workspace_size(int B, int T, int S, int d_model, int H, int H_kv,
                                   int d_k, int d_v);

/*
 * mha_sublayer_fwd -- the multi-head attention sublayer, asynchronous on
 * `stream`:
 *
 *     q = x W_q + b_q,  k = mem W_k + b_k,  v = mem W_v + b_v
 *     head_i = Attention(q_i, k_g, v_g),  g = i / (H / H_kv)
 *     out = Concat(head_1, ..., head_H) W_o + b_o
 *
 * (trishampatil.com, "Multi-Head Attention" and "The Output Projection W^O";
 * aicassindra.com, "A faithful layer in code").  Head i of a projection is its
 * columns [i d, (i + 1) d), so q, k, v are the [B, L, heads, d] layout of
 * mha_fwd_ex and the attention output is already the concatenation.
 *
 * x      [B, T, d_model] queries' token vectors
 * mem    [B, S, d_model] keys' and values' token vectors (encoder memory for
 *        cross-attention), or NULL for self-attention (then S must equal T)
 * out    [B, T, d_model]
 * w_q    [d_model, H d_k],   w_k [d_model, H_kv d_k],   w_v [d_model, H_kv d_v],
 * w_o    [H d_v, d_model];   b_* their output widths, each may be NULL
 * mask_kind, key_lengths, scale: as for mha_fwd (masks apply to the
 *        attention step; key_lengths [B] on the device)
 * workspace  device memory of at least mha_sublayer_workspace_size(...) bytes,
 *        256-byte aligned, owned by the caller, not overlapping any argument;
 *        the call uses it until the enqueued work has run
 * All matrices bf16 (dtype MHA_DTYPE_BF16), 16-byte aligned; d_model, H d_k,
 * H_kv d_k, H_kv d_v, H d_v multiples of 8; d_k = d_v in {64, 128} (the
 * attention step's rule).  Validation covers every step before anything is
 * enqueued.  Ownership and errors as for mha_fwd.
 */
int mha_sublayer_fwd(const void *x, const void *mem, void *out,
                     const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                     const void *b_q, const void *b_k, const void *b_v, const void *b_o,
                     int B, int T, int S, int d_model, int H, int H_kv, int d_k, int d_v,
                     int mask_kind, const int32_t *key_lengths, float scale, int dtype,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * mha_sublayer_fwd_static -- mha_sublayer_fwd without a caller workspace.
 *
 * The pages have no counterpart: this is an interface convenience.  For
 * callers that cannot provide device memory for the intermediates (hosts whose
 * device memory is budgeted up front and must not allocate on their serving
 * path, C callers without a device allocator of their own).  The library uses
 * its own static device scratch of 64 MiB per device (reserved when the
 * library's device code is loaded); nothing is allocated per call.  Shapes
 * whose mha_sublayer_workspace_size exceeds 64 MiB return MHA_ERR_UNSUPPORTED
 * (use mha_sublayer_fwd).  The first call on a device looks the scratch up
 * (make that call before any stream capture).  All calls on a device share the
 * one scratch: calls that overlap in time, on other streams or threads, race
 * on it and must be serialised by the caller.  Arguments and errors otherwise
 * as for mha_sublayer_fwd.
 */
int mha_sublayer_fwd_static(const void *x, const void *mem, void *out,
                            const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                            const void *b_q, const void *b_k, const void *b_v, const void *b_o,
                            int B, int T, int S, int d_model, int H, int H_kv, int d_k, int d_v,
                            int mask_kind, const int32_t *key_lengths, float scale, int dtype,
                            void *stream);

/* Bytes of device workspace mha_bwd needs: two fp32 values per query row
   (the row's log-sum-exp and D = dout . out), 256-byte aligned parts; 0 for
   an empty problem. */
size_t mha_bwd_workspace_size(int B, int H, int Lq);

/*
 * mha_bwd -- gradients of a loss through the attention, for training,
 * asynchronous on `stream`.
 *
 * The pages train the model end to end, every position of the target
 * sequence at once under the causal mask, with the gradients flowing back
 * through every layer (trishampatil.com, "Training (Teacher Forcing +
 * Masking)"); they print no backward formulas.  These are the derivatives of
 * the forward of mha_fwd_ex by the chain rule: with w_ij the softmax weights
 * of the allowed keys,
 *
 *     dP_ij = dout_i . v_j,   D_i = dout_i . out_i,   dS_ij = w_ij (dP_ij - D_i)
 *     dq_i = scale sum_j dS_ij k_j,   dk_j = scale sum_i dS_ij q_i,
 *     dv_j = sum_i w_ij dout_i
 *
 * (with shared key/value heads, dk and dv of head g sum over the query heads
 * that read g).  Rows whose output is fixed at +0 (query padding, no allowed
 * key) have dq = 0 and contribute nothing; keys no row may read get dk = dv = 0.
 *
 * q, k, v, layout, mask_kind, key_lengths, scale, dtype, H_kv: as for
 *                      mha_fwd_ex, the values of the forward call
 * out                  that call's output (for D_i)
 * dout                 dL/dout, out's shape and layout
 * dq, dk, dv           results: the shapes and layout of q, k and v, dtype
 *                      `dtype`; overwritten entirely
 * workspace            device memory of at least mha_bwd_workspace_size(B, H,
 *                      Lq) bytes, 256-byte aligned, caller-owned; its contents
 *                      need not be initialised and are scratch afterwards
 *
 * All pointers are device pointers, 16-byte aligned; the gradients overlap no
 * input, each other, the workspace or key_lengths.  Calls that share a
 * workspace must not overlap in time.  Shapes, dtypes and masks supported
 * and the errors returned are those of mha_fwd_ex; MHA_ERR_INVALID_ARGUMENT
 * also for a missing or too small workspace.  The weights are recomputed
 * from the inputs (nothing is kept from the forward call but `out`).
 */
int mha_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
            void *dq, void *dk, void *dv, int B, int H, int H_kv, int Lq, int Lk, int d_k,
            int d_v, int layout, int mask_kind, const int32_t *key_lengths, float scale,
            int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * mha_bwd_lse -- mha_bwd given the forward pass's row statistics `lse` (from
 * mha_fwd_lse with the same arguments): the weights are formed from them, so
 * no statistics pass recomputes the scores (6 products per allowed (query,
 * key) pair instead of 8 on the tensor cores); only D = dout . out is formed
 * first.  lse: device float[B, H, Lq], 4-byte aligned, read only, must not
 * overlap dq, dk, dv or the workspace; NULL is MHA_ERR_INVALID_ARGUMENT
 * unless B*H*Lq == 0.  The fp32 path and the single-tile bf16 path (d = 64,
 * Lq, Lk <= 128: one fused kernel that forms the statistics itself) read it
 * not.  Every other argument, the workspace and the errors are those of
 * mha_bwd.
 */
int mha_bwd_lse(const void *q, const void *k, const void *v, const void *out, const void *dout,
                const float *lse, void *dq, void *dk, void *dv, int B, int H, int H_kv, int Lq,
                int Lk, int d_k, int d_v, int layout, int mask_kind, const int32_t *key_lengths,
                float scale, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* Which kernel mha_fwd would launch for these arguments:
   0 = none (empty problem), 1 = fp32 CUDA-core kernel, 2 = packed
   short-sequence tensor-core kernel (Lq, Lk <= 128), 3 = long-sequence
   tensor-core kernel, 4 = zero fill (Lk == 0), 5 = few-query tensor-core
   kernel (decoding steps: at most 16 query rows per key/value head, mask
   NONE, KEY_PADDING and/or CAUSAL_TAIL, Lk > 128 or d = 128); negative =
   -(mha_status) for arguments mha_fwd would reject.  Host only, launches
   nothing. */
int mha_fwd_path(int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind, int dtype);

/* The same for mha_fwd_ex with H_kv key/value heads (mha_fwd_path is this
   with H_kv = H); an H_kv that does not divide H gives
   -MHA_ERR_INVALID_ARGUMENT. */
int mha_fwd_path_ex(int B, int H, int H_kv, int Lq, int Lk, int d_k, int d_v, int mask_kind,
                    int dtype);

/* Static text for a status code. */
const char *mha_status_string(int status);

/* Reads and clears the device-side status word that kernels set when a
   bounded wait runs out (MHA_ERR_TIMEOUT).  Synchronises `stream`.  Returns
   MHA_OK, MHA_ERR_TIMEOUT, or MHA_ERR_CUDA if the read itself failed. */
int mha_debug_status(void *stream);

/*
 * mha_debug_set_wait -- test hook for the kernels' give-up path (the pages
 * have no counterpart).
 *
 * Every wait inside the tensor-core kernels is bounded: after `limit_ns` of
 * wall time (default 2 s) the waiting warp gives up, the CTA lets the copies
 * and products it has in flight finish, frees its tensor memory and records
 * MHA_ERR_TIMEOUT in the status word that mha_debug_status() reads.  This call
 * sets that limit for the calls enqueued after it (0 restores the default)
 * and, for tests, `stall` bits that make a kernel wait on a barrier nothing
 * signals, so the give-up path runs without any fault:
 *   1  packed short-sequence kernel: the MMA issuer stalls before its first
 *      product;
 *   2  long-sequence kernel: the MMA issuer stalls before its third key
 *      tile, with products and copies in flight.
 * The output of a stalled call is undefined.  Process-wide setting; not for
 * use while other threads enqueue work.  Returns MHA_ERR_INVALID_ARGUMENT for
 * unknown stall bits.
 */
int mha_debug_set_wait(unsigned long long limit_ns, int stall);

/* Library version as 10000*major + 100*minor + patch. */
int mha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_H */
