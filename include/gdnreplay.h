/*
 * gdnreplay.h -- C ABI of libgdnreplay: ReplaySSM-style verify / accept / flush
 * of Gated DeltaNet (GDN) recurrent state under speculative decoding, as
 * hand-written CUDA kernels for sm_103a (GB300).
 *
 * Method ("The inference stack behind OCRia", LlamaIndex engineering blog,
 * section "Making speculative verification cheaper"): the recurrent state of a
 * GDN layer is large, so moving it per token (and restoring it after a rejected
 * draft) costs HBM traffic.  ReplaySSM keeps, per sequence, a checkpoint of the
 * state and a short buffer of the inputs committed since; the draft's outputs
 * come from replaying that buffer and the draft over the checkpoint, the
 * checkpoint itself is rewritten only when the buffer is flushed, and a
 * rejection only moves the buffer's length back.  Drafts are accepted up to the
 * first rejected token ("Inference Engineering", chapter 5, speculative
 * decoding).
 *
 * Recurrence (the gated delta rule of "Gated Delta Networks", Yang, Kautz &
 * Hatamizadeh, ICLR 2025; the blog names GDN without printing it), per
 * sequence b and head h, with state S of shape [d_v, d_k]:
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t (scale q_t),   alpha_t = exp(g_t),   scale = 1/sqrt(d_k)
 * q and k arrive L2-normalised; the kernels do not re-normalise them.
 *
 * Layouts (row-major, innermost last; every tensor dense and contiguous):
 *   state      fp32     [n_slot, H, dv, dk]   checkpoint per state slot
 *   state_idx  int32    [B]                   slot of batch row b; NULL = identity
 *                                             (slots must be distinct, < n_slot)
 *   buf_k      in_dtype [n_slot, H, cap, dk]  committed (and staged draft) keys
 *   buf_v      in_dtype [n_slot, H, cap, dv]
 *   buf_g      fp32     [n_slot, H, cap]      log-decay g (alpha = exp(g)), g <= 0
 *   buf_beta   fp32     [n_slot, H, cap]
 *   buf_len    int32    [n_slot]              committed tokens in the buffer
 *   q, k       in_dtype [B, T, H, dk]         draft block
 *   v          in_dtype [B, T, H, dv]
 *   g, beta    fp32     [B, T, H]
 *   out        fp32     [B, T, H, dv]
 *   accepted   int32    [B]                   accepted draft tokens, 0..T
 *   status     int32    [1]                   device word; kernels OR fault bits in
 * in_dtype is bf16 (GDN_DTYPE_BF16) or fp32 (GDN_DTYPE_F32).
 * All pointers except dims are DEVICE pointers; dims is a host pointer read
 * during the call only.
 *
 * Ownership and concurrency: the caller owns every buffer.  The library never
 * allocates, frees or synchronises, and keeps no global state; each call only
 * enqueues kernels on the given stream and returns.  Calls on one layer's
 * buffers must be stream-ordered.
 *
 * Errors: 0 on success.  Host-side validation returns a negative code before
 * anything is launched (see GDN_ERR_*).  Faults found on the device (a bad
 * accepted count, no room in the buffer, a corrupt length) never trap: the
 * kernel ORs a GDN_STATUS_* bit into *status, skips the affected sequence and
 * continues.  Read *status after the stream has completed.
 */
#ifndef GDNREPLAY_H
#define GDNREPLAY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;

#define GDN_DTYPE_BF16 0
#define GDN_DTYPE_F32  1

#define GDN_OK            0
#define GDN_ERR_NULL     -1   /* a required pointer is NULL */
#define GDN_ERR_DIMS     -2   /* unsupported or inconsistent dims */
#define GDN_ERR_DTYPE    -3   /* in_dtype is not GDN_DTYPE_BF16 / GDN_DTYPE_F32 */
#define GDN_ERR_LAUNCH   -4   /* the CUDA launch itself failed (cudaGetLastError) */

#define GDN_STATUS_BAD_ACCEPT 1   /* accepted[b] outside [0, T]; b left unchanged */
#define GDN_STATUS_NO_ROOM    2   /* verify: buf_len + T > cap; b skipped */
#define GDN_STATUS_BAD_LEN    4   /* buf_len outside [0, cap] (accept: len + p > cap); b skipped */
#define GDN_STATUS_BAD_SLOT   8   /* state_idx[b] outside [0, n_slot); b skipped */
#define GDN_STATUS_TIMEOUT   16   /* a bounded on-chip wait expired; the (b, h) unit was skipped.
                                     While this bit is set in *status, gdn_replay_flush and
                                     gdn_replay_accept_fold reset no buffer length, so the
                                     buffer of a unit whose fold gave up is kept.  The units
                                     folded by the same call then hold their new checkpoint
                                     and still their buffer length: after a TIMEOUT in a flush
                                     or a fused step, restore the layer (checkpoint, buffer,
                                     lengths) from a saved copy before the next verify */
#define GDN_STATUS_DRAIN     32   /* after an expired wait, the wait for that unit's own copies and
                                     tensor-core operations expired too; its tensor memory was
                                     released anyway (a kernel never hangs), so no result of the
                                     call may be trusted */

/* Bits of gdn_replay_dims.flags.  Every other bit must be 0 (GDN_ERR_DIMS otherwise). */
#define GDN_FLAG_TEST_EXPIRE  1   /* test only: every tensor-core kernel takes its wait-expiry exit
                                     at its first bounded wait, before it has issued any copy or
                                     tensor-core operation, so the GDN_STATUS_TIMEOUT path runs
                                     without anything in flight.  Never set in production. */

/* Kernel families (gdn_replay_kernel_family). */
#define GDN_FAMILY_TCGEN05   1    /* tcgen05 tensor-core kernels: dk = dv = 128, bf16 inputs, T <= 16,
                                     cap <= 80 */
#define GDN_FAMILY_PERTOKEN  2    /* per-token CUDA-core kernels: every other valid shape */

typedef struct {
    int32_t B;          /* batch rows (sequences) in this call, >= 0 */
    int32_t H;          /* heads, >= 1 */
    int32_t dk;         /* key/query head dim: 64 or 128 */
    int32_t dv;         /* value head dim (state rows): 64 or 128 */
    int32_t T;          /* draft block length, 1..64 */
    int32_t cap;        /* buffer slots per (slot, head), T <= cap <= 256; the per-token
                           kernels hold the buffer and the draft in shared memory, so
                           (cap (dk + dv + 2) + T dk) 4 bytes must fit in 227 KB (else
                           GDN_ERR_DIMS), with cap + T in place of cap for
                           gdn_replay_verify_fold: at dk = dv = 128, T = 16, cap <= 217,
                           and <= 201 for the fused step */
    int32_t threshold;  /* flush when buf_len >= threshold, 1..cap */
    int32_t n_slot;     /* state / buffer slots, >= B */
    int32_t in_dtype;   /* GDN_DTYPE_BF16 or GDN_DTYPE_F32 */
    float   scale;      /* query scale, normally 1/sqrt(dk) */
    int32_t flags;      /* GDN_FLAG_* bits; 0 in production */
} gdn_replay_dims;

/*
 * gdn_replay_verify -- the verify pass of the blog's section "Making
 * speculative verification cheaper": draft outputs from the checkpoint replayed
 * with the buffered inputs.
 * For every b with slot s = state_idx[b] and len = buf_len[s], and every head:
 * start from state[s,h], replay the len committed tokens of the buffer, then
 * the T draft tokens, writing o_t = S_t (scale q_t) to out[b,t,h,:] for each
 * draft token.  The checkpoint and buf_len are NOT written.  The draft
 * (k, v, g, beta) is copied into buffer slots [len, len+T) so that accepting p
 * tokens later is a pure length update.  If len < 0 or len + T > cap the
 * sequence is skipped (out untouched) and GDN_STATUS_NO_ROOM is set.
 */
int gdn_replay_verify(const gdn_replay_dims *dims,
                      const float *state, const int32_t *state_idx,
                      void *buf_k, void *buf_v, float *buf_g, float *buf_beta,
                      const int32_t *buf_len,
                      const void *q, const void *k, const void *v,
                      const float *g, const float *beta,
                      float *out, int32_t *status, cudaStream_t stream);

/*
 * gdn_replay_accept -- rollback and commit as a length update only (blog, same
 * section: no state is restored): buf_len[s] += accepted[b] when
 * 0 <= accepted[b] <= T and the result fits in cap; rejected draft tokens stay
 * in the buffer as stale slots that the next verify overwrites.  Otherwise a
 * status bit is set and buf_len[s] is left unchanged.  Writes only buf_len.
 */
int gdn_replay_accept(const gdn_replay_dims *dims, int32_t *buf_len,
                      const int32_t *state_idx, const int32_t *accepted,
                      int32_t *status, cudaStream_t stream);

/*
 * gdn_replay_flush -- the periodic rewrite of the checkpoint (blog, same
 * section).  For every b whose len = buf_len[s] satisfies
 * len >= threshold, or len > 0 when force != 0: replay the len buffered tokens
 * onto state[s,h] for every head, write the result back in place (fp32) and set
 * buf_len[s] = 0.  Other sequences are left bit-identical.  A len outside
 * [0, cap] sets GDN_STATUS_BAD_LEN and skips the sequence.
 */
int gdn_replay_flush(const gdn_replay_dims *dims, float *state,
                     const int32_t *state_idx,
                     const void *buf_k, const void *buf_v,
                     const float *buf_g, const float *buf_beta,
                     int32_t *buf_len, int32_t force, int32_t *status,
                     cudaStream_t stream);

/*
 * Lazy flush -- the periodic flush folded into the next verify, so the
 * checkpoint of a flushed sequence is read once instead of twice (the fusion
 * the blog's section "Avoiding unnecessary memory transfers" argues for, applied
 * to the flush of "Making speculative verification cheaper").  A decode step is
 *     gdn_replay_verify_fold(...);  gdn_replay_accept_fold(...);
 * and is equivalent to  gdn_replay_flush(force = 0); gdn_replay_verify; gdn_replay_accept.
 *
 * gdn_replay_verify_fold -- as gdn_replay_verify, except that a sequence whose
 * len = buf_len[s] is >= threshold first has its len buffered tokens folded into
 * state[s,h] (written in place, fp32) and its draft staged at buffer slots
 * [0, T) instead of [len, len+T).  Outputs are those of verify after that fold.
 * buf_len is NOT written (every head of a sequence reads the same len); the
 * following gdn_replay_accept_fold applies the reset.  Requires
 * threshold - 1 + T <= cap; lengths before the call may reach threshold - 1 + T.
 */
int gdn_replay_verify_fold(const gdn_replay_dims *dims,
                           float *state, const int32_t *state_idx,
                           void *buf_k, void *buf_v, float *buf_g, float *buf_beta,
                           const int32_t *buf_len,
                           const void *q, const void *k, const void *v,
                           const float *g, const float *beta,
                           float *out, int32_t *status, cudaStream_t stream);

/*
 * gdn_replay_accept_fold -- the accept that follows gdn_replay_verify_fold:
 * buf_len[s] = (len >= threshold ? 0 : len) + accepted[b], with the checks of
 * gdn_replay_accept.  Writes only buf_len.
 */
int gdn_replay_accept_fold(const gdn_replay_dims *dims, int32_t *buf_len,
                           const int32_t *state_idx, const int32_t *accepted,
                           int32_t *status, cudaStream_t stream);

/*
 * gdn_replay_kernel_family -- which kernels a verify / flush / verify_fold call with
 * these dims launches: GDN_FAMILY_TCGEN05 or GDN_FAMILY_PERTOKEN, or a negative
 * GDN_ERR_* code for dims the calls would reject.  Host only; launches nothing.  A
 * call whose dims select GDN_FAMILY_TCGEN05 never runs the per-token kernels: if the
 * tensor-core launch cannot be prepared (for example the driver's tensor-map encoder
 * cannot be resolved) the call returns GDN_ERR_LAUNCH.
 */
int gdn_replay_kernel_family(const gdn_replay_dims *dims);

/* Human-readable text for a GDN_ERR_* code (static storage). */
const char *gdn_replay_strerror(int code);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gdn_replay_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDNREPLAY_H */
