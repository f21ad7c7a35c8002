/*
 * gdnnonreplay.h -- C ABI of the non-replay baseline for Gated DeltaNet state
 * under speculative decoding: the data movement that checkpoint + buffer replay
 * avoids, built so that the two can be measured side by side on one GPU.
 *
 * Source: "The inference stack behind OCRia" (LlamaIndex engineering blog),
 * section "Making speculative verification cheaper": a recurrent layer has no
 * per-token cache to truncate, so without a checkpoint and a buffer a rejected
 * draft forces the state back to the accepted prefix, and restoring it moves a
 * lot of data.  Here the state is always current: the verify stores the state
 * after every draft token, and the accept restores by copying the snapshot of
 * the accepted prefix over the state (prefix acceptance: "Inference
 * Engineering", chapter 5, speculative decoding).
 *
 * Recurrence (Gated Delta Networks, ICLR 2025), per (sequence, head), S of
 * shape [d_v, d_k]:  S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 * o_t = S_t (scale q_t), alpha_t = exp(g_t); computed in fp32.
 *
 * Dimensions: gdn_replay_dims (gdnreplay.h) with B >= 0, H >= 1, d_k, d_v in
 * {64, 128}, 1 <= T <= 64, n_slot >= 0, in_dtype GDN_DTYPE_BF16 or
 * GDN_DTYPE_F32, flags 0; cap and threshold are not used (there is no buffer).
 * Without state_idx, n_slot >= B.  B = 0 returns GDN_OK without touching any
 * pointer.
 *
 * Layouts (row-major, last index contiguous; all device pointers, caller-owned;
 * the library allocates nothing, never synchronises and keeps no state):
 *   state    fp32     [n_slot, H, d_v, d_k]   verify reads it; accept writes it
 *   state_idx int32   [B] slot of batch row b, or NULL for the identity
 *   q, k     in_dtype [B, T, H, d_k];  v in_dtype [B, T, H, d_v]
 *   g, beta  fp32     [B, T, H]
 *   out      fp32     [B, T, H, d_v]
 *   snap     fp32     [B, H, T, d_v, d_k]     state after draft token t (t = 0..T-1)
 *   accepted int32    [B];  status int32 [1], OR-ed, never cleared by the library
 * state and snap must be 16-byte aligned.
 *
 * Errors: the host checks return GDN_ERR_NULL / GDN_ERR_DIMS / GDN_ERR_DTYPE
 * before any launch and GDN_ERR_LAUNCH when the launch fails.  On the device a
 * slot outside [0, n_slot) sets GDN_STATUS_BAD_SLOT and an accepted count
 * outside [0, T] sets GDN_STATUS_BAD_ACCEPT; the row is skipped (nothing of it
 * written); no kernel traps.
 */
#ifndef GDNNONREPLAY_H
#define GDNNONREPLAY_H

#include "gdnreplay.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Outputs of the draft block from the current state, and every intermediate
 * state stored in snap.  Writes out and snap; never writes state. */
int gdn_nonreplay_verify(const gdn_replay_dims *dims, const float *state, const int32_t *state_idx,
                         const void *q, const void *k, const void *v, const float *g, const float *beta,
                         float *out, float *snap, int32_t *status, cudaStream_t stream);

/* Restore by copy: state[slot_b] = snap[b, :, p_b - 1] for p_b in [1, T]; p_b = 0
 * (everything rejected) leaves the state.  Writes only state. */
int gdn_nonreplay_accept(const gdn_replay_dims *dims, float *state, const int32_t *state_idx,
                         const float *snap, const int32_t *accepted, int32_t *status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNNONREPLAY_H */
