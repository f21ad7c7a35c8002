// replay_common.h -- definitions shared by the CUDA translation units of
// libgdnreplay (not part of the public ABI; see include/gdnreplay.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdnreplay.h"

namespace gdn {

// Arguments of one verify or flush launch (device pointers, layouts of gdnreplay.h).
struct ReplayArgs {
    const float *state_in;      // verify: checkpoint (read)
    float *state_out;           // flush: checkpoint (read + write)
    const int32_t *state_idx;
    void *buf_k, *buf_v;
    float *buf_g, *buf_beta;
    const int32_t *buf_len;
    const void *q, *k, *v;
    const float *g, *beta;
    float *out;
    int32_t *status;
    int B, H, T, cap, threshold, force, n_slot;
    float scale;
};

// Internal status bit: a bounded wait in a tensor-core kernel gave up (the
// affected unit is skipped; nothing hangs).
constexpr int32_t kStatusTimeout = GDN_STATUS_TIMEOUT;

// Tensor-core path (gdn_replay_tc.cu).  Each returns GDN_OK when it launched,
// GDN_ERR_LAUNCH on a launch failure, and 1 when the shape is not one it
// handles (the caller then uses the per-token kernels).
// fold = true: units whose buffer reached the threshold also write the checkpoint
// after their buffered tokens and stage the draft at buffer slot 0.
int tc_verify(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s, bool fold);
int tc_flush(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s);

}  // namespace gdn
