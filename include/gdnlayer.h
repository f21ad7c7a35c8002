/*
 * gdnlayer.h -- C ABI of the two GDN layer steps either side of the recurrence in
 * libgdnreplay (sm_103a): the causal convolution before it, with the same
 * pointer rollback as the recurrent state, and the gated RMSNorm with FP8
 * quantisation after it.  "The inference stack behind OCRia" (LlamaIndex
 * engineering blog), section "Avoiding unnecessary memory transfers", names both
 * among the kernels it fused or sped up ("a faster causal convolution for GDN
 * layers"; "gated RMSNorm followed by FP8 quantisation").  Conventions as in
 * gdnreplay.h: device pointers, a host dims struct read during the call only,
 * no allocation, no synchronisation, no global state, 0 or a negative GDN_ERR_*
 * code from host validation, device faults OR-ed into a status word.
 */
#ifndef GDNLAYER_H
#define GDNLAYER_H

#include <stdint.h>

#include "gdnreplay.h"

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_CONV_ACT_NONE 0
#define GDN_CONV_ACT_SILU 1

/*
 * Causal depthwise convolution under speculative decoding.
 *
 * For channel c and kernel width W (the short convolution GDN layers apply to
 * q, k and v before the recurrence; "Gated Delta Networks", ICLR 2025):
 *     y_t[c] = act( bias[c] + sum_{j=0}^{W-1} weight[c][j] * x_{t-(W-1)+j}[c] ).
 * For a draft block x_0 .. x_{T-1}, the inputs x_{-(W-1)} .. x_{-1} are the last
 * W-1 committed inputs of the sequence.  They sit in a ring of `cap` positions
 * per slot with write position ring_pos[s]: the window is positions
 * ring_pos-W+1 .. ring_pos-1 (mod cap).  gdn_conv_verify emits y for the draft and
 * stages the draft inputs at positions ring_pos .. ring_pos+T-1 (mod cap), so
 * that accepting p tokens (gdn_conv_accept) only advances ring_pos by p: rejected
 * draft inputs are never part of a later window, and no window is restored (the
 * rollback of the blog's section "Making speculative verification cheaper").
 *
 * Layouts (row-major, innermost last, dense):
 *   ring      in_dtype  [n_slot, cap, D]
 *   ring_pos  int32     [n_slot]        0 <= ring_pos < cap
 *   state_idx int32     [B]             slot of sequence b; NULL = identity
 *   x         in_dtype  [B, T, D]       draft inputs (pre-convolution)
 *   weight    fp32      [D, W]          weight[c][W-1] multiplies the current input; 16-byte aligned
 *   bias      fp32      [D] or NULL (16-byte aligned)
 *   y         out_dtype [B, T, D]
 *   accepted  int32     [B]             0..T
 * Arithmetic in fp32; a bf16 y is rounded to nearest even once at the end.
 * Device faults: GDN_STATUS_BAD_SLOT (state_idx[b] out of range),
 * GDN_STATUS_BAD_LEN (ring_pos out of range), GDN_STATUS_BAD_ACCEPT; the
 * sequence is skipped.
 */
typedef struct {
    int32_t B;          /* sequences in this call, >= 0 */
    int32_t D;          /* channels, a multiple of 8 */
    int32_t W;          /* kernel width, 1..4 */
    int32_t T;          /* draft block length, 1..64 */
    int32_t cap;        /* ring positions per slot, W - 1 + T <= cap <= 4096 */
    int32_t n_slot;     /* ring slots, >= B */
    int32_t act;        /* GDN_CONV_ACT_NONE or GDN_CONV_ACT_SILU */
    int32_t in_dtype;   /* GDN_DTYPE_BF16 or GDN_DTYPE_F32 (x and the ring) */
    int32_t out_dtype;  /* GDN_DTYPE_BF16 or GDN_DTYPE_F32 (y) */
} gdn_conv_dims;

int gdn_conv_verify(const gdn_conv_dims *dims, void *ring, const int32_t *ring_pos,
                    const int32_t *state_idx, const void *x, const float *weight,
                    const float *bias, void *y, int32_t *status, cudaStream_t stream);

/* ring_pos[s] = (ring_pos[s] + accepted[b]) mod cap for 0 <= accepted[b] <= T;
 * otherwise a status bit is set and ring_pos[s] is left unchanged.  Writes only
 * ring_pos. */
int gdn_conv_accept(const gdn_conv_dims *dims, int32_t *ring_pos, const int32_t *state_idx,
                    const int32_t *accepted, int32_t *status, cudaStream_t stream);

/*
 * Gated RMSNorm fused with FP8 (E4M3) quantisation, per row of d values:
 *     r = 1 / sqrt(mean_i(o_i^2) + eps),   y_i = o_i * r * weight[i] * silu(z_i),
 *     q_i = E4M3(y_i * inv_scale)   (round to nearest even, saturated to +-448).
 * The GDN output o (e.g. gdn_replay_verify's out, viewed as [B*T*H, dv]) is
 * normalised per head and gated by z; inv_scale is a static per-tensor scale
 * (dequantise with q * (1 / inv_scale)).  E4M3: 1 sign, 4 exponent and 3 mantissa
 * bits ("Inference Engineering", chapter 5, number formats), bias 7, no infinity.
 *   o      fp32     [rows, d]
 *   z      z_dtype  [rows, d]   GDN_DTYPE_BF16 or GDN_DTYPE_F32
 *   weight fp32     [d]
 *   q      uint8    [rows, d]   E4M3 codes
 * d is 64, 128 or 256.  Arithmetic in fp32; the code is taken from the fp32 value.
 */
int gdn_gated_rmsnorm_fp8(int32_t rows, int32_t d, const float *o, const void *z, int32_t z_dtype,
                          const float *weight, float eps, float inv_scale, uint8_t *q,
                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNLAYER_H */
