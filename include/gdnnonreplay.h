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

/* Size of the snapshot area inside the library that gdn_nonreplay_step_static uses:
 * it serves steps with B * H * T * d_v * d_k * 4 <= this many bytes (e.g. 512 snapshots
 * at d = 128: B = 2, H = 16, T = 16).  Every GPU that loads the library holds it until
 * the process exits. */
#define GDN_NONREPLAY_STATIC_SNAP_BYTES (32u << 20)

/* One baseline step (gdn_nonreplay_verify, then gdn_nonreplay_accept) that allocates
 * nothing: the snapshots go to a fixed area inside the library instead of a caller
 * buffer.  The paper has no counterpart; this exists for callers that can pass tensors
 * but cannot call cudaMalloc -- a plugin inside a serving engine whose device memory is
 * reserved up front by the engine's own allocator and offers the plugin no allocation
 * hook, or a latency-bound loop where cudaMalloc's implicit device synchronisation is
 * not allowed.  Inputs and outputs are those of the two calls it replaces: state
 * (updated in place), state_idx, q, k, v, g, beta, accepted, out, status.
 *
 * A step larger than GDN_NONREPLAY_STATIC_SNAP_BYTES of snapshots returns GDN_ERR_DIMS
 * before anything is launched.  Every call looks up the area's device address in the
 * current context (host-side, no synchronisation; the first lookup in a context loads
 * the library's device code there, so make the first call before any stream capture).
 * Every call shares the one area and leaves its snapshots there; nothing in it needs
 * clearing (the verify writes every snapshot the accept reads), but calls whose work
 * overlaps on the GPU -- on different streams, or from different threads -- race on it
 * and must be serialised by the caller. */
int gdn_nonreplay_step_static(const gdn_replay_dims *dims, float *state, const int32_t *state_idx,
                              const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const int32_t *accepted, float *out, int32_t *status,
                              cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNNONREPLAY_H */
