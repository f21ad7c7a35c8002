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
    int fold_class;             // 0: all units; 1: only the units that do not fold, launched
                                // beside the fold launch
    int flags;                  // gdn_replay_dims.flags (GDN_FLAG_TEST_EXPIRE)
};

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialisation and waits (griddepcontrol.wait) before its first
// read of global memory another kernel may have written.  All but the verify kernel
// then let the next kernel on the stream start its launch and prologue
// (launch_dependents); the verify kernel does so only before its epilogue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Internal status bit: a bounded wait in a tensor-core kernel gave up (the
// affected unit is skipped; nothing hangs).
constexpr int32_t kStatusTimeout = GDN_STATUS_TIMEOUT;

// Tensor-core path (gdn_replay_tc.cu): d_k = d_v = 128, bf16 inputs, T <= 16,
// cap <= 80 (tc_shape).  Each returns GDN_OK when it launched, GDN_ERR_LAUNCH when
// the launch (or the tensor map it needs) failed, and 1 only when the shape is not
// one it handles (the caller then uses the per-token kernels).
bool tc_shape(const gdn_replay_dims *d);
int tc_verify(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s);
int tc_flush(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s);
// The fused step: the folding sequences (persistent fold kernel, which then verifies
// their drafts) and, beside it, the effective-query verify of every other sequence.
int tc_verify_fold(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s);

}  // namespace gdn
