// gdn_replay_tc.cu -- tensor-core (tcgen05) verify / flush kernels of
// libgdnreplay for sm_103a, for d_k = d_v = 128 and bf16 inputs.
//
// Chunked form.  For one (sequence, head) replaying C tokens (the committed
// buffer, then the draft block) from the checkpoint S0, with G_t the running
// sum of the log-decays g and gamma_t = e^{G_t}, the gated delta rule
// ("Gated Delta Networks", ICLR 2025) unrolls into the chunkwise form of
// "Parallelizing Linear Transformers with the Delta Rule over Sequence
// Length" (NeurIPS 2024):
//   u_t = beta_t (v_t - gamma_t S0 k_t) - sum_{s<t} beta_t e^{G_t-G_s} (k_t.k_s) u_s
//   o_t = scale (gamma_t S0 q_t + sum_{s<=t} e^{G_t-G_s} (q_t.k_s) u_s)
//   S_C = gamma_C S0 + sum_s e^{G_C-G_s} u_s k_s^T
// The d_v x d_k contractions (S0 [K;Q]^T, and for the flush U^T K) run on the
// tensor cores; the forward substitution is row-local (one thread per state
// row, row i = TMEM lane i) and only exponentiates G_t - G_s <= 0.
//
// Data movement: the checkpoint tile (64 KB fp32) arrives by TMA with 128-byte
// swizzle, which is the K-major layout tcgen05 reads directly.  Keys and
// queries are bf16 in HBM; threads widen them into a swizzled fp32 tile.  The
// accumulators live in TMEM and are read back with tcgen05.ld.  Every wait is
// bounded: on expiry the unit is skipped, a status bit is set, and the kernel
// still waits (bounded) for its own copies and MMAs before freeing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "replay_common.h"

namespace gdn {
namespace {

constexpr int kThreads = 128;               // one thread per state row / TMEM lane
constexpr uint32_t kWaitLimit = 1u << 21;   // mbarrier polls before giving up
constexpr int kTmemCols = 256;

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(saddr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_tile_l2(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {   // 16-byte multiples
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {   // one full warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)),
                 "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // the allocating warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(src))
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_wait() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tcgen05 descriptor version 1).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor: fp32 accumulator, A/B format `fmt` (tf32 = 2, bf16 = 1),
// both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_mn(int fmt, int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &raw, float *f) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(p[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

__host__ __device__ inline int round16(int x) { return (x + 15) & ~15; }

// Three bf16 terms whose sum is x exactly (for normal-range x): each rounding
// to bf16 keeps the next 8-9 significant bits of what is left.
__device__ __forceinline__ void split3(float x, __nv_bfloat16 &h, __nv_bfloat16 &m, __nv_bfloat16 &l) {
    h = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(h);
    m = __float2bfloat16_rn(r1);
    l = __float2bfloat16_rn(r1 - __bfloat162float(m));
}
// Two bf16 terms whose sum is x to a relative 2^-16.
__device__ __forceinline__ void split2(float x, __nv_bfloat16 &h, __nv_bfloat16 &l) {
    h = __float2bfloat16_rn(x);
    l = __float2bfloat16_rn(x - __bfloat162float(h));
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// ---------------------------------------------------------------------------
// Forward substitution in blocks of 16 tokens (one state row per thread).
//   u_t = beta_t (v_t - gamma_t P_t) - sum_{s<t} A[t][s] u_s,   t < C
// and, when Mt is given, the draft sums o[t2] = sum_s M[t2][s] u_s.
// Earlier blocks' u live in shared memory (this thread's column of sU), so the
// cross-block update is a rolled loop and the unrolled code is one 16 x 16
// triangle: the instruction stream stays small enough to be cached.
//   At  [>= CP rows][LDT]  A transposed (At[s][t] = A[t][s]); zeros at s >= t
//   Mt  [>= CP rows][16]   M transposed (Mt[s][t2] = M[t2][s]); zeros past p
//   sV  [C][128] bf16      value rows;  sU [C][128] fp32 receives u
//   P   TMEM columns [0, C) of this thread's lane (S0 k_t)
// Tokens t >= C get u = 0 (their coefficient entries may be unset).
__device__ __forceinline__ void blocked_solve(int C, int tid, uint32_t lane_base, const float *At, int LDT,
                                              const float *Mt, const __nv_bfloat16 *sV, float *sU,
                                              const float *sBeta, const float *sGam, float (&o)[16])
{
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = 0.f;
    const int nb = (C + 15) >> 4;
#pragma unroll 1
    for (int kb = 0; kb < nb; ++kb) {
        const int t0 = kb * 16;
        float pc[16], r[16];
        tmem_ld16(lane_base + t0, pc);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = t0 + j;
            const float vt = t < C ? __bfloat162float(sV[static_cast<size_t>(t) * 128 + tid]) : 0.f;
            r[j] = t < C ? sBeta[t] * (vt - sGam[t] * pc[j]) : 0.f;
        }
        // contributions of the earlier blocks
#pragma unroll 2
        for (int s = 0; s < t0; ++s) {
            const float us = sU[static_cast<size_t>(s) * 128 + tid];
            const float4 *a4 = reinterpret_cast<const float4 *>(At + static_cast<size_t>(s) * LDT + t0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = a4[q];
                r[4 * q] = fmaf(-x.x, us, r[4 * q]);
                r[4 * q + 1] = fmaf(-x.y, us, r[4 * q + 1]);
                r[4 * q + 2] = fmaf(-x.z, us, r[4 * q + 2]);
                r[4 * q + 3] = fmaf(-x.w, us, r[4 * q + 3]);
            }
        }
        // the 16 x 16 triangle of this block, right-looking
#pragma unroll
        for (int jp = 0; jp < 16; ++jp) {
            const float uj = (t0 + jp < C) ? r[jp] : 0.f;
            r[jp] = uj;
            const float4 *a4 = reinterpret_cast<const float4 *>(At + static_cast<size_t>(t0 + jp) * LDT + t0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = a4[q];
                if (4 * q > jp) r[4 * q] = fmaf(-x.x, uj, r[4 * q]);
                if (4 * q + 1 > jp) r[4 * q + 1] = fmaf(-x.y, uj, r[4 * q + 1]);
                if (4 * q + 2 > jp) r[4 * q + 2] = fmaf(-x.z, uj, r[4 * q + 2]);
                if (4 * q + 3 > jp) r[4 * q + 3] = fmaf(-x.w, uj, r[4 * q + 3]);
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (t0 + j < C) sU[static_cast<size_t>(t0 + j) * 128 + tid] = r[j];
        if (Mt) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 *m4 = reinterpret_cast<const float4 *>(Mt + static_cast<size_t>(t0 + j) * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = m4[q];
                    o[4 * q] = fmaf(x.x, r[j], o[4 * q]);
                    o[4 * q + 1] = fmaf(x.y, r[j], o[4 * q + 1]);
                    o[4 * q + 2] = fmaf(x.z, r[j], o[4 * q + 2]);
                    o[4 * q + 3] = fmaf(x.w, r[j], o[4 * q + 3]);
                }
            }
        }
    }
}

// P[i][C + t2] for t2 < 16 from two 16-column TMEM chunks starting at C & ~15: the
// uniform rotation by C & 15 keeps every register index static.
__device__ __forceinline__ void pq_rotate(float (&pq)[2][16], int sh, float (&out)[16]) {
    float p[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) { p[i] = pq[0][i]; p[16 + i] = pq[1][i]; }
#pragma unroll
    for (int bit = 0; bit < 4; ++bit) {
        const int k = 1 << bit;
        if (sh & k) {
#pragma unroll
            for (int i = 0; i < 32; ++i) p[i] = i + k < 32 ? p[i + k] : 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = p[i];
}

// Shared-memory plan of the verify kernel (bytes from the 1024-aligned base):
//   [0, 64K)          S0 tile (fp32, 4 sub-tiles of 128 rows x 128 B, TMA).  After the
//                     MMAs, in a folding unit: U~ as three bf16 tiles [0, 48K) and K^T
//                     (bf16) [48K, 64K) for the fold MMA, then the new state for the
//                     TMA store.
//   [64K, 64K + SB)   [K;Q] fp32 tile, 4 sub-tiles of NP rows x 128 B, plus slack so an
//                     M=128 operand may read past row NP.  After the MMAs: coefficient
//                     matrices (row stride CP+4) followed by the S0 q columns.
//   then: 4 mbarriers, TMEM slot, flags, and G (hi, lo), beta, gamma per token, each
//   array padded to a multiple of 16 tokens so it can be read as float4.
// cmax = most tokens one unit replays: cap (verify), cap + T (verify with fold, where a
// full buffer is replayed together with the draft).  The dynamic shared memory base is
// the start of the CTA's shared window (no static shared variables), so it is 1024-byte
// aligned; the kernel checks this and, if it ever fails, reports it in the status word
// and skips the unit.
__host__ __device__ inline int verify_sb_bytes(int cmax, int T) { return (3 * round16(cmax + T) + 128) * 128; }
__host__ __device__ inline int verify_smem_bytes(int cmax, int T) {
    return 65536 + verify_sb_bytes(cmax, T) + 64 + 20 * round16(cmax);
}

// FOLD = false: gdn_replay_verify.  FOLD = true: gdn_replay_verify_fold -- a unit whose
// buffer has reached the threshold also writes the checkpoint after its buffered
// tokens (the flush, done here instead of in a separate pass over the state) and
// stages the draft at buffer slot 0.
template <int CMAX, bool FOLD>
__global__ void __launch_bounds__(kThreads, 2)
verify_tc_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int T = a.T, H = a.H, cap = a.cap;
    const int cmax = FOLD ? cap + T : cap;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (saddr(smem_raw) & 1023u) {           // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) atomicOr(a.status, kStatusTimeout);
        return;
    }
    uint8_t *base = smem_raw;
    uint8_t *sA = base;
    uint8_t *sB = base + 65536;
    uint8_t *sm = sB + verify_sb_bytes(cmax, T);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);            // TMA, K.K MMA, P MMA, fold MMA
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 32);
    int *flag = reinterpret_cast<int *>(sm + 36);
    const int GS = round16(cmax);                                 // per-token array stride (16-B rows)
    float *sGh = reinterpret_cast<float *>(sm + 64);
    float *sGl = sGh + GS;
    float *sBeta = sGl + GS;
    float *sGam = sBeta + GS;
    float *sFold = sGam + GS;                                     // e^{G_{len-1} - G_s}, folding units
    uint8_t *sU = sA;                                             // fold: 3 x 16 KB
    uint8_t *sKt = sA + 49152;                                    // fold: 16 KB

    // prologue that touches no global memory: overlaps the previous kernel
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_release();

    const int slot = a.state_idx ? a.state_idx[b] : b;
    const int len = (slot >= 0 && slot < a.n_slot) ? a.buf_len[slot] : 0;
    const bool fold = FOLD && len >= a.threshold && len <= cap;
    int bad = 0;
    if (slot < 0 || slot >= a.n_slot) bad = GDN_STATUS_BAD_SLOT;
    else if (len < 0 || (!fold && len + T > cap)) bad = len < 0 || len > cap ? GDN_STATUS_BAD_LEN : GDN_STATUS_NO_ROOM;
    // fold_class 2: only the folding units; the others belong to the launch that follows
    const bool other_class = a.fold_class == 2 && !fold;
    if (bad || other_class) {                                     // uniform across the CTA
        if (bad && tid == 0 && h == 0) atomicOr(a.status, bad);
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    const int C = len + T;                   // replayed tokens: buffer, then draft
    const int NP = round16(C + T);           // rows of the [K;Q] operand
    const int CP = round16(C);               // key columns of the K.K / Q.K product
    const int row0 = fold ? 0 : len;         // buffer slot of draft token 0

    const size_t unit = static_cast<size_t>(slot) * H + h;
    const int ytile = static_cast<int>(unit) * 128;
    if (tid == 0) {                                               // checkpoint tile by TMA
        mbar_expect_tx(&bar[0], 65536);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) tma_load_2d(sA + kb * 16384, &tm_state, kb * 32, ytile, &bar[0]);
    }

    // ---- the unit that will run one wave later (CTA index + prefetch_stride): its
    //      checkpoint tile, buffer rows and draft rows are prefetched into L2 now, so
    //      the DRAM reads of that wave overlap this wave's compute
    if (a.prefetch_stride > 0 && warp == 1) {
        const int lane = tid & 31;
        const int nxt = b * gridDim.x + h + a.prefetch_stride;
        if (nxt < static_cast<int>(gridDim.x * gridDim.y)) {
            const int nb = nxt / gridDim.x, nh = nxt % gridDim.x;
            const int ns = a.state_idx ? a.state_idx[nb] : nb;
            if (ns >= 0 && ns < a.n_slot) {
                const int nlen = min(max(a.buf_len[ns], 0), cap);
                const size_t nunit = static_cast<size_t>(ns) * H + nh;
                if (lane < 4) prefetch_tile_l2(&tm_state, lane * 32, static_cast<int>(nunit) * 128);
                if (lane == 4 && nlen > 0)
                    prefetch_l2(reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + nunit * cap * 128, nlen * 256);
                if (lane == 5 && nlen > 0)
                    prefetch_l2(reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + nunit * cap * 128, nlen * 256);
                const size_t nrow0 = (static_cast<size_t>(nb) * T * H + nh) * 128;
                for (int r = lane; r < 3 * T; r += 32) {           // draft k, q, v rows (256 B each)
                    const void *base3 = r < T ? a.k : r < 2 * T ? a.q : a.v;
                    prefetch_l2(reinterpret_cast<const __nv_bfloat16 *>(base3) + nrow0 +
                                    static_cast<size_t>(r % T) * H * 128, 256);
                }
            }
        }
    }

    // ---- every global load of this unit, issued back to back (one memory latency)
    const __nv_bfloat16 *bk = reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
    const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
    const size_t drow0 = (static_cast<size_t>(b) * T * H + h) * 128;   // draft token 0 of (b, h)
    const size_t dstride = static_cast<size_t>(H) * 128;
    const __nv_bfloat16 *dk = reinterpret_cast<const __nv_bfloat16 *>(a.k) + drow0;
    const __nv_bfloat16 *dq = reinterpret_cast<const __nv_bfloat16 *>(a.q) + drow0;
    const __nv_bfloat16 *dv = reinterpret_cast<const __nv_bfloat16 *>(a.v) + drow0;
    __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(a.buf_k) + (unit * cap + row0) * 128;
    __nv_bfloat16 *wv = reinterpret_cast<__nv_bfloat16 *>(a.buf_v) + (unit * cap + row0) * 128;
    constexpr int NV = (CMAX + 16) * 16 / kThreads;               // 16-byte vectors of [K;Q] per thread
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C + T) {
            const __nv_bfloat16 *src = r < len ? bk + static_cast<size_t>(r) * 128
                                     : r < C   ? dk + static_cast<size_t>(r - len) * dstride
                                               : dq + static_cast<size_t>(r - C) * dstride;
            raw[i] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
        }
    }
    // value rows as 16-byte vectors (moved through shared memory once the S0 tile is free)
    constexpr int NVV = CMAX * 16 / kThreads;
    uint4 vload[NVV];
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) {
            const __nv_bfloat16 *src = r < len ? bv + static_cast<size_t>(r) * 128
                                               : dv + static_cast<size_t>(r - len) * dstride;
            vload[i] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
        }
    }
    // fold: the draft keys are re-staged at slot 0 after every buffer read is done
    uint4 kdraft[2];
    if (fold) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
            if (r < T) kdraft[i] = __ldg(reinterpret_cast<const uint4 *>(dk + static_cast<size_t>(r) * dstride) + c);
        }
    }
    float gq[2] = {0.f, 0.f}, bq[2] = {0.f, 0.f};                 // gates of tokens lane, lane + 32 (warp 0)
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = (tid & 31) + 32 * i;
            if (t < C) {
                if (t < len) {
                    gq[i] = a.buf_g[unit * cap + t];
                    bq[i] = a.buf_beta[unit * cap + t];
                } else {
                    const size_t gi = (static_cast<size_t>(b) * T + (t - len)) * H + h;
                    gq[i] = a.g[gi];
                    bq[i] = a.beta[gi];
                }
            }
        }
    }
    // ---- widen [K;Q] into the swizzled fp32 tile; draft keys into the buffer (no fold)
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C + T) {
            if (!fold && r >= len && r < C) reinterpret_cast<uint4 *>(wk + static_cast<size_t>(r - len) * 128)[c] = raw[i];
            float f[8];
            bf16x8_to_f32(raw[i], f);
            uint8_t *tile = sB + (c >> 2) * NP * 128;
            const int ch = (c & 3) * 2;
            *reinterpret_cast<float4 *>(tile + sw128(r, ch)) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(tile + sw128(r, ch + 1)) = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    if (warp == 0) {
        // running log-decay G_t = sum_{s<=t} g_s as a compensated pair (hi + lo): a
        // Kogge-Stone scan with two-sum steps over tokens lane and lane + 32
        const int lane = tid & 31;
        float hi[2], lo[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            hi[i] = gq[i];
            lo[i] = 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float h2 = __shfl_up_sync(0xffffffffu, hi[i], off);
                const float l2 = __shfl_up_sync(0xffffffffu, lo[i], off);
                if (lane >= off) {
                    const float s1 = hi[i] + h2, bp = s1 - hi[i];
                    lo[i] += l2 + ((hi[i] - (s1 - bp)) + (h2 - bp));
                    hi[i] = s1;
                }
            }
        }
        const float ch = __shfl_sync(0xffffffffu, hi[0], 31), cl = __shfl_sync(0xffffffffu, lo[0], 31);
        {
            const float s1 = hi[1] + ch, bp = s1 - hi[1];
            lo[1] += cl + ((hi[1] - (s1 - bp)) + (ch - bp));
            hi[1] = s1;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = lane + 32 * i;
            if (t < C) {
                sGh[t] = hi[i];
                sGl[t] = lo[i];
                sGam[t] = __expf(hi[i] + lo[i]);
                sBeta[t] = bq[i];
                if (!fold && t >= len) {
                    a.buf_g[unit * cap + t] = gq[i];
                    a.buf_beta[unit * cap + t] = bq[i];
                }
            }
        }
    }
    fence_proxy_async();                      // generic writes of the [K;Q] tile -> async proxy
    __syncthreads();
    if (tid == 0) {
        if (mbar_wait(&bar[0], 0)) {
            tc_fence_after();
            const uint32_t idP = idesc_mn(2, 128, NP), idK = idesc_mn(2, 128, CP);
            const uint32_t a0 = saddr(sA), b0 = saddr(sB);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {                      // [K;Q] K^T first (coefficients)
                const uint64_t d = desc_sw128(b0 + (ks >> 2) * NP * 128 + (ks & 3) * 32);
                mma_tf32(tmem + NP, d, d, idK, ks > 0);
            }
            mma_commit(&bar[1]);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {                      // P = S0 [K;Q]^T, K = 128 in steps of 8
                const uint32_t off = (ks & 3) * 32;
                mma_tf32(tmem, desc_sw128(a0 + (ks >> 2) * 16384 + off),
                         desc_sw128(b0 + (ks >> 2) * NP * 128 + off), idP, ks > 0);
            }
            mma_commit(&bar[2]);
        } else {
            *flag = 1;
        }
    }
    __syncthreads();
    bool ok = *flag == 0;
    if (ok) ok = mbar_wait(&bar[1], 0);
    if (__syncthreads_or(!ok)) {
        // give up on this unit: wait (bounded) for in-flight copies / MMAs, report, free TMEM
        if (tid == 0) {
            mbar_wait(&bar[0], 0);
            if (*flag == 0) {
                mbar_wait(&bar[1], 0);
                mbar_wait(&bar[2], 0);
            }
            atomicOr(a.status, kStatusTimeout);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);

    // ---- coefficient rows from K.K / Q.K (TMEM lane = token), kept in registers until
    //      the P MMA has finished reading the [K;Q] tile they will be written over:
    //      A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s) for s < t, M[t'][s] = e^{G_p-G_s} (q_t'.k_s)
    //      for s <= p = len + t'
    float m[CMAX / 16][16];
    {
        const bool is_q = tid >= C;
        const int p = tid >= C + T ? C - 1 : is_q ? len + (tid - C) : tid;   // position of this row's token
        const float gh = sGh[p], gl = sGl[p];
        const float scl = is_q ? 1.f : sBeta[p];
        const int lim = tid >= C + T ? 0 : is_q ? min(p + 1, C) : tid;   // columns s < lim are used
#pragma unroll
        for (int cb = 0; cb < CMAX / 16; ++cb) {
            const int c0 = cb * 16;
            if (c0 >= CP) break;
            float kq[16];
            tmem_ld16(lane_base + NP + c0, kq);
            float gs[16], ls[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 x = *reinterpret_cast<const float4 *>(sGh + c0 + 4 * j);
                const float4 y = *reinterpret_cast<const float4 *>(sGl + c0 + 4 * j);
                gs[4 * j] = x.x; gs[4 * j + 1] = x.y; gs[4 * j + 2] = x.z; gs[4 * j + 3] = x.w;
                ls[4 * j] = y.x; ls[4 * j + 1] = y.y; ls[4 * j + 2] = y.z; ls[4 * j + 3] = y.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float e = __expf((gh - gs[j]) + (gl - ls[j]));
                m[cb][j] = (c0 + j < lim) ? scl * e * kq[j] : 0.f;
            }
        }
    }
    // ---- the P MMA has landed: S0 q columns, fold K^T, then the coefficient rows
    ok = mbar_wait(&bar[2], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            mbar_wait(&bar[2], 0);
            atomicOr(a.status, kStatusTimeout);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    tc_fence_after();
    float pq[2][16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {                                 // columns [C & ~15, +32) hold S0 q
        const int c0 = (C & ~15) + 16 * i;
        if (c0 < C + T) tmem_ld16(lane_base + c0, pq[i]);
    }
    if (fold) {                                                   // K^T (bf16) from the fp32 key tile
        const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
        const uint8_t *colbase = sB + (tid >> 5) * NP * 128 + (tid & 3) * 4;
#pragma unroll
        for (int c8 = 0; c8 < CMAX / 8; ++c8) {
            if (c8 * 8 >= round16(len)) break;                   // the MMA reads round16(len) tokens
            __nv_bfloat16 kk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int s = c8 * 8 + j;
                kk[j] = s < len ? __float2bfloat16_rn(*reinterpret_cast<const float *>(
                                      colbase + sw128(s, (tid & 31) >> 2)))
                                : zero;
            }
            *reinterpret_cast<uint4 *>(sKt + sw128(tid, c8)) =
                make_uint4(pack2(kk[0], kk[1]), pack2(kk[2], kk[3]), pack2(kk[4], kk[5]), pack2(kk[6], kk[7]));
        }
    }
    // park the value rows in the free S0 tile; once every thread has its loads back
    // (the barrier), no read of the old buffer is outstanding and the draft (k, v, g,
    // beta) can be staged into slots row0 .. row0 + T - 1
    __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(sA);   // [C][128] bf16
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) reinterpret_cast<uint4 *>(sV + static_cast<size_t>(r) * 128)[c] = vload[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r >= len && r < C) reinterpret_cast<uint4 *>(wv + static_cast<size_t>(r - len) * 128)[c] = vload[i];
    }
    if (fold) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
            if (r < T) reinterpret_cast<uint4 *>(wk + static_cast<size_t>(r) * 128)[c] = kdraft[i];
        }
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int t = (tid & 31) + 32 * i;
                if (t >= len && t < C) {
                    a.buf_g[unit * cap + (t - len)] = gq[i];
                    a.buf_beta[unit * cap + (t - len)] = bq[i];
                }
            }
        }
    }
    if (fold && warp == 0) {                                      // fold factors, shared by all rows
        const float gh = sGh[len - 1], gl = sGl[len - 1];
        for (int t = tid; t < round16(len); t += 32)
            sFold[t] = t < len ? __expf((gh - sGh[t]) + (gl - sGl[t])) : 0.f;
    }
    __syncthreads();                                              // [K;Q] tile no longer read
    // value rows sit in sA [0, 16K); the transposed coefficient matrices go to
    // sA [16K, 36K) (K^T of a fold stays at sA [48K, 64K)) and u to the [K;Q] tile
    float *Mt = reinterpret_cast<float *>(sA + 16384);            // [CP][16]
    float *At = reinterpret_cast<float *>(sA + 20480);            // [CP][CP]
    float *sUf = reinterpret_cast<float *>(sB);                   // [C][128]
    if (tid < C + T) {
        float *dst = tid < C ? At + tid : Mt + (tid - C);
        const int ld = tid < C ? CP : 16;
#pragma unroll
        for (int cb = 0; cb < CMAX / 16; ++cb) {
            if (cb * 16 >= CP) break;
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[static_cast<size_t>(cb * 16 + j) * ld] = m[cb][j];
        }
    }
    __syncthreads();

    // ---- forward substitution and draft sums, then o_t = scale (gamma_p S0 q_t + sum_s M[t][s] u_s)
    float o[16];
    blocked_solve(C, tid, lane_base, At, CP, Mt, sV, sUf, sBeta, sGam, o);
    {
        float pqr[16];
        pq_rotate(pq, C & 15, pqr);
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2) {
            if (t2 < T) {
                const int p = len + t2;
                a.out[((static_cast<size_t>(b) * T + t2) * H + h) * 128 + tid] =
                    a.scale * (sGam[p] * pqr[t2] + o[t2]);
            }
        }
    }
    // ---- fold: U~_s = e^{G_{len-1} - G_s} u_s (s < len) as three bf16 tiles, then
    //      D = U~^T K on the tensor cores
    if (fold) {
        __syncthreads();                                          // value rows, coefficients read
#pragma unroll 1
        for (int c8 = 0; c8 < round16(len) / 8; ++c8) {          // the MMA reads round16(len) tokens
            __nv_bfloat16 hh[8], mm[8], ll[8];
            const float4 f0 = *reinterpret_cast<const float4 *>(sFold + c8 * 8);
            const float4 f1 = *reinterpret_cast<const float4 *>(sFold + c8 * 8 + 4);
            const float fs[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = c8 * 8 + j;
                const float ut = t < len ? sUf[static_cast<size_t>(t) * 128 + tid] : 0.f;
                split3(fs[j] * ut, hh[j], mm[j], ll[j]);
            }
            const uint32_t off = sw128(tid, c8);
            *reinterpret_cast<uint4 *>(sU + off) =
                make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
            *reinterpret_cast<uint4 *>(sU + 16384 + off) =
                make_uint4(pack2(mm[0], mm[1]), pack2(mm[2], mm[3]), pack2(mm[4], mm[5]), pack2(mm[6], mm[7]));
            *reinterpret_cast<uint4 *>(sU + 32768 + off) =
                make_uint4(pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idF = idesc_mn(1, 128, 128);
            const uint32_t u0 = saddr(sU), kt0 = saddr(sKt);
            const int ksteps = round16(len) / 16;
            for (int sp = 0; sp < 3; ++sp)
                for (int ks = 0; ks < ksteps; ++ks)
                    mma_bf16(tmem, desc_sw128(u0 + sp * 16384 + ks * 32), desc_sw128(kt0 + ks * 32), idF,
                             (sp | ks) != 0);
            mma_commit(&bar[3]);
        }
    }
    if (fold) {
        // ---- new checkpoint S_len = gamma_{len-1} S0 + D, written over the S0 tile and
        //      stored by TMA; S0 row `tid` is read again from global memory (L2)
        const float4 *s0 = reinterpret_cast<const float4 *>(a.state_in + (unit * 128 + tid) * 128);
        float4 x[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) x[q] = s0[q];
        ok = mbar_wait(&bar[3], 0);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                mbar_wait(&bar[3], 0);
                atomicOr(a.status, kStatusTimeout);
            }
            tc_fence_before();
            __syncthreads();
            if (warp == 0) tmem_dealloc(tmem, kTmemCols);
            return;
        }
        tc_fence_after();
        const float gL = sGam[len - 1];
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float d[16];
            tmem_ld16(lane_base + c0, d);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int col = c0 + 4 * q;
                float4 y = x[col >> 2];
                y.x = fmaf(gL, y.x, d[4 * q]);
                y.y = fmaf(gL, y.y, d[4 * q + 1]);
                y.z = fmaf(gL, y.z, d[4 * q + 2]);
                y.w = fmaf(gL, y.w, d[4 * q + 3]);
                *reinterpret_cast<float4 *>(sA + (col >> 5) * 16384 + sw128(tid, (col & 31) >> 2)) = y;
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) tma_store_2d(&tm_state, kb * 32, ytile, sA + kb * 16384);
            tma_store_commit_and_wait();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Verify by effective queries (no fold; T <= 16, C = len + T <= CMAX).
//
// The chunked form gives u = (I + A)^{-1} r with r_s = beta_s (v_s - gamma_s S0 k_s),
// A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s) (s < t), and the draft outputs
// o_t2 = scale (gamma_p S0 q_t2 + sum_s M[t2][s] u_s) with
// M[t2][s] = e^{G_p-G_s} (q_t2.k_s) (s <= p = len + t2).  With W = M (I + A)^{-1}
// (T x C) the sum is sum_s W[t2][s] r_s, so
//   o_t2 = scale (S0 qe_t2 + ve_t2),
//   qe_t2 = gamma_p q_t2 - sum_s W[t2][s] beta_s gamma_s k_s,
//   ve_t2 = sum_s W[t2][s] beta_s v_s.
// The checkpoint enters a single M = 128, N = 16 contraction; everything else
// depends on the tokens only.  W comes from the back substitution
// W[t2][s] = M[t2][s] - sum_{s' > s} W[t2][s'] A[s'][s], one warp per four draft
// rows and one lane per two token columns; qe and ve are bf16 contractions of the
// key and value rows (read as MN-major operands, no transpose) with W beta gamma
// and W beta split into two bf16 terms each (relative error 2^-16).
// The checkpoint is prefetched into L2 at the start and streamed through two
// 16 KB buffers in quarters of 32 columns once the token work is done.
//
// Shared-memory plan (bytes from the 1024-aligned base), NPA = round16(CMAX + 16):
//   [0, 2 SUBK)          [K;Q] rows, bf16, 2 sub-tiles (d_k halves) of NPA rows x 128 B
//   [OFF_V, +2 SUBV)     value rows, bf16, 2 sub-tiles of CMAX rows x 128 B
//   [OFF_A, +CMAX^2 4)   A, fp32, row-major [CMAX][CMAX]
//   [OFF_M, +16 CMAX 4)  M, fp32, row-major [16][CMAX]
//   [OFF_W, +8K)         W beta gamma and W beta as 2 + 2 bf16 tiles [16][64]; later
//                        qe as fp32 [16][128] (4 sub-tiles of 16 rows x 128 B)
//   [0, 32K)             after the token contractions: two checkpoint quarter buffers
//   [OFF_S, ...)         8 mbarriers, TMEM slot, flag, then G (hi, lo), beta, gamma
// An M = 128 operand starting in the [K;Q] tile reads on past its NPA rows; those
// rows only feed accumulator lanes that are never read.
constexpr int kTmemColsEq = 128;
template <int CMAX> struct EqPlan {
    static constexpr int NPA = (CMAX + 16 + 15) & ~15;
    static constexpr int SUBK = NPA * 128;
    static constexpr int SUBV = CMAX * 128;
    static constexpr int OFF_V = 2 * SUBK;
    static constexpr int OFF_A = OFF_V + 2 * SUBV;
    static constexpr int OFF_M = OFF_A + CMAX * CMAX * 4;
    static constexpr int OFF_W = (OFF_M + 16 * CMAX * 4 + 1023) & ~1023;
    static constexpr int OFF_S = OFF_W + 8192;
    static constexpr int BYTES = OFF_S + 128 + 16 * CMAX;
    static_assert(OFF_W >= 32768, "the quarter buffers must not reach the qe tile");
    static_assert(SUBK + 16384 <= BYTES, "M = 128 operand reads stay inside the allocation");
    static_assert(CMAX % 16 == 0 && CMAX <= 64, "token columns: at most two per lane");
    static_assert((SUBK % 1024) == 0 && (OFF_V % 1024) == 0 && (SUBV % 1024) == 0, "swizzle atoms");
};

// MN-major operand, 128-byte swizzle: 64-element atoms along M/N `lbo` bytes apart,
// 8-row groups along K 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t lbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
constexpr uint32_t kIdescMnMajorA = 1u << 15;

template <int CMAX>
__global__ void __launch_bounds__(kThreads, 4)
verify_eq_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    using P = EqPlan<CMAX>;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, H = a.H, cap = a.cap;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (saddr(smem_raw) & 1023u) {           // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) atomicOr(a.status, kStatusTimeout);
        return;
    }
    uint8_t *sKQ = smem_raw;
    uint8_t *sV = smem_raw + P::OFF_V;
    float *sAm = reinterpret_cast<float *>(smem_raw + P::OFF_A);
    float *sMm = reinterpret_cast<float *>(smem_raw + P::OFF_M);
    uint8_t *sW = smem_raw + P::OFF_W;
    uint8_t *sQe = sW;
    uint8_t *sm = smem_raw + P::OFF_S;
    // 0, 1: checkpoint buffers (TMA); 2: K.K; 3: qe, ve; 4..7: checkpoint quarter MMAs
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 64);
    int *flag = reinterpret_cast<int *>(sm + 68);
    float *sGh = reinterpret_cast<float *>(sm + 128);
    float *sGl = sGh + CMAX;
    float *sBeta = sGl + CMAX;
    float *sGam = sBeta + CMAX;
    constexpr int COL_Q = CMAX, COL_V = CMAX + 16, COL_O = CMAX + 32;   // TMEM columns

    if (tid == 0) {                                               // prologue: no global memory
#pragma unroll
        for (int i = 0; i < 8; ++i) mbar_init(&bar[i], 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemColsEq);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // fold_class 1: the units that do not fold, in a launch that runs beside the fold
    // launch preceding it and must not wait for it (every CTA of that launch has
    // waited for the earlier kernels before letting this one start); CTA (0, 0) waits
    // for it at the end instead, so the next kernel observes both launches complete.
    // It reports the length errors of every sequence (the fold launch skips them).
    const bool split = a.fold_class == 1;
    const bool waiter = split && blockIdx.x == 0 && blockIdx.y == 0;
    if (!split) pdl_wait();

    const int slot = a.state_idx ? a.state_idx[b] : b;
    const int len = (slot >= 0 && slot < a.n_slot) ? a.buf_len[slot] : 0;
    const bool other_class = split && len >= a.threshold && len <= cap;   // the fold launch's unit
    int bad = 0;
    if (slot < 0 || slot >= a.n_slot) bad = GDN_STATUS_BAD_SLOT;
    else if (len < 0 || len > cap) bad = GDN_STATUS_BAD_LEN;
    else if (!other_class && len + T > cap) bad = GDN_STATUS_NO_ROOM;
    pdl_release();                                                // every length of this CTA is read
    auto finish = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemColsEq);
        if (waiter) pdl_wait();
    };
    if (bad || other_class) {                                     // uniform across the CTA
        if (bad && tid == 0 && h == 0) atomicOr(a.status, bad);
        finish();
        return;
    }
    const int C = len + T;
    const int CP = round16(C);
    const size_t unit = static_cast<size_t>(slot) * H + h;
    const int ytile = static_cast<int>(unit) * 128;

    // ---- every global load of this unit, issued back to back (the checkpoint, needed
    //      last, is prefetched into L2 once these rows are in, so they come first)
    const __nv_bfloat16 *bk = reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
    const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
    const size_t drow0 = (static_cast<size_t>(b) * T * H + h) * 128;
    const size_t dstride = static_cast<size_t>(H) * 128;
    const __nv_bfloat16 *dk = reinterpret_cast<const __nv_bfloat16 *>(a.k) + drow0;
    const __nv_bfloat16 *dq = reinterpret_cast<const __nv_bfloat16 *>(a.q) + drow0;
    const __nv_bfloat16 *dv = reinterpret_cast<const __nv_bfloat16 *>(a.v) + drow0;
    __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(a.buf_k) + (unit * cap + len) * 128;
    __nv_bfloat16 *wv = reinterpret_cast<__nv_bfloat16 *>(a.buf_v) + (unit * cap + len) * 128;
    constexpr int NV = P::NPA * 16 / kThreads;                   // 16-byte vectors of [K;Q] per thread
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < C + T) {
            const __nv_bfloat16 *src = r < len ? bk + static_cast<size_t>(r) * 128
                                     : r < C   ? dk + static_cast<size_t>(r - len) * dstride
                                               : dq + static_cast<size_t>(r - C) * dstride;
            raw[i] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
        }
    }
    constexpr int NVV = CMAX * 16 / kThreads;
    uint4 vload[NVV];
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        vload[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < C) {
            const __nv_bfloat16 *src = r < len ? bv + static_cast<size_t>(r) * 128
                                               : dv + static_cast<size_t>(r - len) * dstride;
            vload[i] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
        }
    }
    float gq[2] = {0.f, 0.f}, bq[2] = {0.f, 0.f};
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = lane + 32 * i;
            if (t < C) {
                if (t < len) {
                    gq[i] = a.buf_g[unit * cap + t];
                    bq[i] = a.buf_beta[unit * cap + t];
                } else {
                    const size_t gi = (static_cast<size_t>(b) * T + (t - len)) * H + h;
                    gq[i] = a.g[gi];
                    bq[i] = a.beta[gi];
                }
            }
        }
    }
    // ---- rows into the swizzled bf16 tiles (zeros past the last token); the draft
    //      keys and values into the buffer (slots len .. len + T - 1, never read here)
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        *reinterpret_cast<uint4 *>(sKQ + (c >> 3) * P::SUBK + sw128(r, c & 7)) = raw[i];
        if (r >= len && r < C) reinterpret_cast<uint4 *>(wk + static_cast<size_t>(r - len) * 128)[c] = raw[i];
    }
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        *reinterpret_cast<uint4 *>(sV + (c >> 3) * P::SUBV + sw128(r, c & 7)) = vload[i];
        if (r >= len && r < C) reinterpret_cast<uint4 *>(wv + static_cast<size_t>(r - len) * 128)[c] = vload[i];
    }
    if (warp == 0) {                                              // compensated scan of g
        float hi[2], lo[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            hi[i] = gq[i];
            lo[i] = 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float h2 = __shfl_up_sync(0xffffffffu, hi[i], off);
                const float l2 = __shfl_up_sync(0xffffffffu, lo[i], off);
                if (lane >= off) {
                    const float s1 = hi[i] + h2, bp = s1 - hi[i];
                    lo[i] += l2 + ((hi[i] - (s1 - bp)) + (h2 - bp));
                    hi[i] = s1;
                }
            }
        }
        const float chh = __shfl_sync(0xffffffffu, hi[0], 31), cll = __shfl_sync(0xffffffffu, lo[0], 31);
        {
            const float s1 = hi[1] + chh, bp = s1 - hi[1];
            lo[1] += cll + ((hi[1] - (s1 - bp)) + (chh - bp));
            hi[1] = s1;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = lane + 32 * i;
            if (t < CMAX) {                                       // zeros past the last token
                const bool live = t < C;
                sGh[t] = live ? hi[i] : 0.f;
                sGl[t] = live ? lo[i] : 0.f;
                sGam[t] = live ? __expf(hi[i] + lo[i]) : 0.f;
                sBeta[t] = live ? bq[i] : 0.f;
                if (live && t >= len) {
                    a.buf_g[unit * cap + t] = gq[i];
                    a.buf_beta[unit * cap + t] = bq[i];
                }
            }
        }
    }
    fence_proxy_async();
    __syncthreads();
    const uint32_t kq0 = saddr(sKQ), v0 = saddr(sV), w0 = saddr(sW), qe0 = saddr(sQe), s00 = saddr(smem_raw);
    if (tid == 0) {                                               // [K;Q] K^T: coefficients
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) prefetch_tile_l2(&tm_state, q * 32, ytile);
        const uint32_t idK = idesc_mn(1, 128, CP);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint64_t d = desc_sw128(kq0 + (ks >> 2) * P::SUBK + (ks & 3) * 32);
            mma_bf16(tmem, d, d, idK, ks > 0);
        }
        mma_commit(&bar[2]);
    }
    // this thread's query column (d_k = tid) for qe, read before the tiles are reused
    float qcol[16];
#pragma unroll
    for (int t2 = 0; t2 < 16; ++t2) {
        const int r = C + t2;                                     // < NPA
        const __nv_bfloat16 x = *reinterpret_cast<const __nv_bfloat16 *>(
            sKQ + (tid >> 6) * P::SUBK + sw128(r, (tid & 63) >> 3) + (tid & 7) * 2);
        qcol[t2] = t2 < T ? __bfloat162float(x) : 0.f;
    }
    bool ok = mbar_wait(&bar[2], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            mbar_wait(&bar[2], 0);
            atomicOr(a.status, kStatusTimeout);
        }
        finish();
        return;
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // ---- coefficient rows: TMEM lane r = row r of [K;Q]; key rows t < C give
    //      A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s) (s < t), query rows C + t2 give
    //      M[t2][s] = e^{G_p-G_s} (q_t2.k_s) (s <= p); rows t2 >= T of M are zero
    if (warp * 32 < C + 16) {                                     // warp-uniform: the loads are collective
        const bool is_q = tid >= C;
        const int t2 = tid - C;
        const bool writes = tid < C + 16;
        const bool live = tid < C + T;
        const int p = !live ? C - 1 : is_q ? len + t2 : tid;
        const float gh = sGh[p], gl = sGl[p];
        const float scl = is_q ? 1.f : sBeta[p];
        const int lim = !live ? 0 : is_q ? min(p + 1, C) : tid;
        float *dst = is_q ? sMm + (writes ? t2 : 0) * CMAX : sAm + tid * CMAX;
#pragma unroll
        for (int cb = 0; cb < CMAX / 16; ++cb) {
            const int c0 = cb * 16;
            float kq[16];
            if (c0 < CP) {
                tmem_ld16(lane_base + c0, kq);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) kq[j] = 0.f;
            }
            float mrow[16];
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                const float4 x = *reinterpret_cast<const float4 *>(sGh + c0 + 4 * j4);
                const float4 y = *reinterpret_cast<const float4 *>(sGl + c0 + 4 * j4);
                const float gs[4] = {x.x, x.y, x.z, x.w}, ls[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int s = c0 + 4 * j4 + j;
                    const float e = __expf((gh - gs[j]) + (gl - ls[j]));
                    mrow[4 * j4 + j] = s < lim ? scl * e * kq[4 * j4 + j] : 0.f;
                }
            }
            if (writes) {
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4)
                    *reinterpret_cast<float4 *>(dst + c0 + 4 * j4) =
                        make_float4(mrow[4 * j4], mrow[4 * j4 + 1], mrow[4 * j4 + 2], mrow[4 * j4 + 3]);
            }
        }
    }
    __syncthreads();
    // ---- W = M (I + A)^{-1}: warp w holds draft rows 4w .. 4w + 3, lane l token columns
    //      l and l + 32; column s is final once every s' > s has been subtracted
    float x0[4], x1[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float *mr = sMm + (4 * warp + i) * CMAX;
        x0[i] = mr[lane];
        x1[i] = lane + 32 < CMAX ? mr[lane + 32] : 0.f;
    }
#pragma unroll 2
    for (int s = C - 1; s >= 0; --s) {
        const float *ar = sAm + s * CMAX;
        const float a0 = ar[lane], a1 = lane + 32 < CMAX ? ar[lane + 32] : 0.f;
        const bool upper = s >= 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float w = __shfl_sync(0xffffffffu, upper ? x1[i] : x0[i], s & 31);
            x0[i] = fmaf(-w, a0, x0[i]);
            x1[i] = fmaf(-w, a1, x1[i]);
        }
    }
    // ---- W beta gamma and W beta as K-major [16][64] tiles, each the sum of two bf16
    //      terms (relative error 2^-16, far below that of the tf32 checkpoint product)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int s = lane + 32 * half;
        if (s < CMAX) {
            const float bs = sBeta[s], bg = bs * sGam[s];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t2 = 4 * warp + i;
                const float w = half ? x1[i] : x0[i];
                __nv_bfloat16 t4[4];
                split2(w * bg, t4[0], t4[1]);
                split2(w * bs, t4[2], t4[3]);
                const uint32_t off = sw128(t2, s >> 3) + (s & 7) * 2;
#pragma unroll
                for (int j = 0; j < 4; ++j) *reinterpret_cast<__nv_bfloat16 *>(sW + j * 2048 + off) = t4[j];
            }
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {                                               // qe^T and ve^T, M = 128, N = 16
        tc_fence_after();
        const uint32_t idQ = idesc_mn(1, 128, 16) | kIdescMnMajorA;
        const int nks = CP / 16;
#pragma unroll
        for (int ks = 0; ks < CMAX / 16; ++ks) {
            if (ks < nks) {
                const uint64_t ak = desc_mn_sw128(kq0 + ks * 2048, P::SUBK);
                const uint64_t av = desc_mn_sw128(v0 + ks * 2048, P::SUBV);
#pragma unroll
                for (int sp = 0; sp < 2; ++sp) {
                    mma_bf16(tmem + COL_Q, ak, desc_sw128(w0 + sp * 2048 + ks * 32), idQ, (sp | ks) != 0);
                    mma_bf16(tmem + COL_V, av, desc_sw128(w0 + (2 + sp) * 2048 + ks * 32), idQ, (sp | ks) != 0);
                }
            }
        }
        mma_commit(&bar[3]);
    }
    ok = mbar_wait(&bar[3], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            mbar_wait(&bar[3], 0);
            atomicOr(a.status, kStatusTimeout);
        }
        finish();
        return;
    }
    tc_fence_after();
    // the token tiles are free: the first two checkpoint quarters come in from L2
    if (tid == 0) {
        fence_proxy_async();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            mbar_expect_tx(&bar[q], 16384);
            tma_load_2d(smem_raw + q * 16384, &tm_state, q * 32, ytile, &bar[q]);
        }
    }
    {                                                             // qe[t2][d_k = tid], fp32 K-major tile
        float dq[16];
        tmem_ld16(lane_base + COL_Q, dq);
        uint8_t *col = sQe + (tid >> 5) * 2048 + (tid & 3) * 4;
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2) {
            const float ge = t2 < T ? sGam[len + t2] : 0.f;
            *reinterpret_cast<float *>(col + sw128(t2, (tid & 31) >> 2)) = fmaf(ge, qcol[t2], -dq[t2]);
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {                                               // O = S0 qe^T, quarter by quarter
        tc_fence_after();
        const uint32_t idO = idesc_mn(2, 128, 16);
        int loads[2] = {1, 1};                                    // TMA loads issued per buffer
        int mmas = 0;                                             // quarters whose MMAs were issued
        bool good = true;
        for (int q = 0; q < 4; ++q) {
            const int buf = q & 1;
            if (!mbar_wait(&bar[buf], q >> 1)) { good = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_tf32(tmem + COL_O, desc_sw128(s00 + buf * 16384 + ks * 32),
                         desc_sw128(qe0 + q * 2048 + ks * 32), idO, (q | ks) != 0);
            mma_commit(&bar[4 + q]);
            mmas = q + 1;
            if (q < 2) {                                          // the buffer is reused once its MMAs are done
                if (!mbar_wait(&bar[4 + q], 0)) { good = false; break; }
                mbar_expect_tx(&bar[buf], 16384);
                tma_load_2d(smem_raw + buf * 16384, &tm_state, (q + 2) * 32, ytile, &bar[buf]);
                ++loads[buf];
            }
        }
        if (!good) {                                              // wait (bounded) for what is in flight
            for (int q = 0; q < mmas; ++q) mbar_wait(&bar[4 + q], 0);
            for (int i = 0; i < 2; ++i) mbar_wait(&bar[i], (loads[i] - 1) & 1);
            *flag = 1;
        }
    }
    __syncthreads();
    ok = *flag == 0;
    if (ok) ok = mbar_wait(&bar[7], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            if (*flag == 0) mbar_wait(&bar[7], 0);
            atomicOr(a.status, kStatusTimeout);
        }
        finish();
        return;
    }
    tc_fence_after();
    {
        float o[16], ve[16];
        tmem_ld16(lane_base + COL_O, o);
        tmem_ld16(lane_base + COL_V, ve);
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2)
            if (t2 < T)
                a.out[((static_cast<size_t>(b) * T + t2) * H + h) * 128 + tid] = a.scale * (o[t2] + ve[t2]);
    }
    finish();
}

// Shared-memory plan of the flush kernel (bytes from the 1024-aligned base):
//   [0, 64K)      S0 tile, fp32, TMA-loaded; rewritten with the new state and TMA-stored
//   [64K, 160K)   S0 as three bf16 tiles (128 x 128 each, 2 sub-tiles of 128 B rows);
//                 after the first MMAs: U~ as three bf16 tiles [64K, 112K), K^T bf16
//                 [112K, 128K) and the coefficient matrix [128K, 160K)
//   [160K, 192K)  K, bf16, 2 sub-tiles of 128 rows x 128 B (rows >= C unused)
//   then: 2 mbarriers, TMEM slot, flag, item count, G (hi, lo), beta, gamma and the
//   fold factors per token, and the list of sequences to flush (kFlushList entries).
constexpr int kFlushList = 1024;
__host__ __device__ inline int flush_smem_bytes(int cap) {
    return 1024 + 196608 + 64 + 20 * round16(cap) + 4 * kFlushList;
}

// Persistent: one CTA per SM.  Every CTA lists the sequences that flush (len >=
// threshold, or len > 0 when forced) and takes (sequence, head) items with a grid
// stride, so only units with work occupy an SM.
template <int CMAX>
__global__ void __launch_bounds__(kThreads, 1)
flush_tc_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = a.H, cap = a.cap;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sS = base;
    uint8_t *sX = base + 65536;
    uint8_t *sU = sX;                                               // 3 x 16 KB after the first MMAs
    uint8_t *sKt = sX + 49152;                                      // 16 KB
    float *sMat = reinterpret_cast<float *>(sX + 65536);            // <= 32 KB
    uint8_t *sK = base + 163840;
    uint8_t *sm = base + 196608;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 16);
    int *flag = reinterpret_cast<int *>(sm + 20);
    int *n_list = reinterpret_cast<int *>(sm + 24);
    const int GS = round16(cap);                                   // per-token array stride (16-B rows)
    float *sGh = reinterpret_cast<float *>(sm + 64);
    float *sGl = sGh + GS;
    float *sBeta = sGl + GS;
    float *sGam = sBeta + GS;
    float *sFold = sGam + GS;
    int *list = reinterpret_cast<int *>(sFold + GS);

    if (tid == 0) {                                                 // prologue: no global memory
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_release();

    uint32_t it = 0;                                                // items done by this CTA
    int *warp_cnt = n_list + 1;                                     // [4] per-warp counts
    for (int b0 = 0; b0 < a.B; b0 += kFlushList) {
        // the list must be identical in every CTA: compact in sequence order with
        // ballots and a prefix over the four warps (no atomics)
        if (tid == 0) *n_list = 0;
        __syncthreads();
        const int bend = min(b0 + kFlushList, a.B);
        for (int g0 = b0; g0 < bend; g0 += kThreads) {
            const int bb = g0 + tid;
            bool f = false;
            if (bb < bend) {
                const int sl = a.state_idx ? a.state_idx[bb] : bb;
                if (sl >= 0 && sl < a.n_slot) {                     // others: reported by the length kernel
                    const int ln = a.buf_len[sl];
                    f = ln >= 0 && ln <= cap && (ln >= a.threshold || (a.force && ln > 0));
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, f);
            if ((tid & 31) == 0) warp_cnt[warp] = __popc(m);
            __syncthreads();
            int base = *n_list;
            for (int w2 = 0; w2 < warp; ++w2) base += warp_cnt[w2];
            if (f) list[base + __popc(m & ((1u << (tid & 31)) - 1u))] = bb;
            __syncthreads();
            if (tid == 0) *n_list += warp_cnt[0] + warp_cnt[1] + warp_cnt[2] + warp_cnt[3];
            __syncthreads();
        }
        const int n_items = *n_list * H;
        for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++it) {
    const int b = list[w / H], h = w % H;
    const int slot = a.state_idx ? a.state_idx[b] : b;
    const int len = a.buf_len[slot];
    const int C = len;
    const int CP = round16(C);
    if (tid == 0) *flag = 0;
    const size_t unit = static_cast<size_t>(slot) * H + h;
    const int y = static_cast<int>(unit) * 128;
    if (tid == 0) {
        mbar_expect_tx(&bar[0], 65536);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) tma_load_2d(sS + kb * 16384, &tm_state, kb * 32, y, &bar[0]);
    }
    // keys of the buffered tokens (bf16, copied as is into the swizzled K tile), the
    // value channel `tid` of every token and the gates: all loads issued back to back
    const __nv_bfloat16 *bk = reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
    const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
    constexpr int NV = CMAX * 16 / kThreads;
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) raw[i] = __ldg(reinterpret_cast<const uint4 *>(bk + static_cast<size_t>(r) * 128) + c);
    }
    constexpr int NVV = CMAX * 16 / kThreads;                       // value rows as 16-byte vectors
    uint4 vload[NVV];
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) vload[i] = __ldg(reinterpret_cast<const uint4 *>(bv + static_cast<size_t>(r) * 128) + c);
    }
    float gq[2] = {0.f, 0.f}, bq[2] = {0.f, 0.f};
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = (tid & 31) + 32 * i;
            if (t < C) {
                gq[i] = a.buf_g[unit * cap + t];
                bq[i] = a.buf_beta[unit * cap + t];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) *reinterpret_cast<uint4 *>(sK + (c >> 3) * 16384 + sw128(r, c & 7)) = raw[i];
    }
    if (warp == 0) {                                                // compensated scan of g (see verify)
        const int lane = tid & 31;
        float hi[2], lo[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            hi[i] = gq[i];
            lo[i] = 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float h2 = __shfl_up_sync(0xffffffffu, hi[i], off);
                const float l2 = __shfl_up_sync(0xffffffffu, lo[i], off);
                if (lane >= off) {
                    const float s1 = hi[i] + h2, bp = s1 - hi[i];
                    lo[i] += l2 + ((hi[i] - (s1 - bp)) + (h2 - bp));
                    hi[i] = s1;
                }
            }
        }
        const float ch = __shfl_sync(0xffffffffu, hi[0], 31), cl = __shfl_sync(0xffffffffu, lo[0], 31);
        {
            const float s1 = hi[1] + ch, bp = s1 - hi[1];
            lo[1] += cl + ((hi[1] - (s1 - bp)) + (ch - bp));
            hi[1] = s1;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = lane + 32 * i;
            if (t < C) {
                sGh[t] = hi[i];
                sGl[t] = lo[i];
                sGam[t] = __expf(hi[i] + lo[i]);
                sBeta[t] = bq[i];
            }
        }
    }
    if (tid == 0 && !mbar_wait(&bar[0], it & 1)) *flag = 1;
    __syncthreads();
    if (*flag) {
        if (tid == 0) {
            mbar_wait(&bar[0], it & 1);
            atomicOr(a.status, kStatusTimeout);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    // ---- S0 row `tid` -> three bf16 tiles (exact split)
    {
        const int r = tid;
#pragma unroll 4
        for (int c8 = 0; c8 < 16; ++c8) {                           // 8 columns per step
            const float4 x0 = *reinterpret_cast<const float4 *>(sS + (c8 >> 2) * 16384 + sw128(r, (c8 & 3) * 2));
            const float4 x1 = *reinterpret_cast<const float4 *>(sS + (c8 >> 2) * 16384 + sw128(r, (c8 & 3) * 2 + 1));
            const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            __nv_bfloat16 hh[8], mm[8], ll[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) split3(xs[j], hh[j], mm[j], ll[j]);
            const uint32_t off = (c8 >> 3) * 16384 + sw128(r, c8 & 7);
            *reinterpret_cast<uint4 *>(sX + off) =
                make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
            *reinterpret_cast<uint4 *>(sX + 32768 + off) =
                make_uint4(pack2(mm[0], mm[1]), pack2(mm[2], mm[3]), pack2(mm[4], mm[5]), pack2(mm[6], mm[7]));
            *reinterpret_cast<uint4 *>(sX + 65536 + off) =
                make_uint4(pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idP = idesc_mn(1, 128, CP);
        const uint32_t x0 = saddr(sX), k0 = saddr(sK);
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {                        // K = 128 in steps of 16 (32 bytes)
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem, desc_sw128(x0 + sp * 32768 + off), desc_sw128(k0 + off), idP, (sp | ks) != 0);
            }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            const uint64_t d = desc_sw128(k0 + off);
            mma_bf16(tmem + CP, d, d, idP, ks > 0);
        }
        mma_commit(&bar[1]);
    }
    bool ok = mbar_wait(&bar[1], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            mbar_wait(&bar[1], 0);
            atomicOr(a.status, kStatusTimeout);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(sX);      // [C][128] in the dead S0 splits
#pragma unroll
    for (int i = 0; i < NVV; ++i) {
        const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
        if (r < C) reinterpret_cast<uint4 *>(sV + static_cast<size_t>(r) * 128)[c] = vload[i];
    }
    // ---- K^T row `tid` (key channel j = tid): k_s[j] for s < CP, zero past C; built
    //      before the key tile is reused for u
    {
        const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
        for (int c8 = 0; c8 < CP / 8; ++c8) {
            __nv_bfloat16 kk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int s2 = c8 * 8 + j;
                kk[j] = s2 < C ? *reinterpret_cast<const __nv_bfloat16 *>(
                                     sK + (tid >> 6) * 16384 + sw128(s2, (tid & 63) >> 3) + (tid & 7) * 2)
                               : zero;
            }
            *reinterpret_cast<uint4 *>(sKt + sw128(tid, c8)) =
                make_uint4(pack2(kk[0], kk[1]), pack2(kk[2], kk[3]), pack2(kk[4], kk[5]), pack2(kk[6], kk[7]));
        }
    }
    // ---- coefficient rows A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s), s < t, stored transposed
    float *At = sMat;                                               // [CP][CP]
    for (int c0 = 0; c0 < CP; c0 += 16) {
        float kq[16];
        tmem_ld16(lane_base + CP + c0, kq);
        if (tid < C) {
            const float gh = sGh[tid], gl = sGl[tid], be = sBeta[tid];
            float gs[16], ls[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 x = *reinterpret_cast<const float4 *>(sGh + c0 + 4 * j);
                const float4 y = *reinterpret_cast<const float4 *>(sGl + c0 + 4 * j);
                gs[4 * j] = x.x; gs[4 * j + 1] = x.y; gs[4 * j + 2] = x.z; gs[4 * j + 3] = x.w;
                ls[4 * j] = y.x; ls[4 * j + 1] = y.y; ls[4 * j + 2] = y.z; ls[4 * j + 3] = y.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float e = __expf((gh - gs[j]) + (gl - ls[j]));
                At[static_cast<size_t>(c0 + j) * CP + tid] = (c0 + j < tid) ? be * e * kq[j] : 0.f;
            }
        }
    }
    if (warp == 0) {                                              // fold factors, shared by all rows
        const float gh = sGh[C - 1], gl = sGl[C - 1];
        for (int t = tid; t < CP; t += 32) sFold[t] = t < C ? __expf((gh - sGh[t]) + (gl - sGl[t])) : 0.f;
    }
    __syncthreads();                                                // key tile read, coefficients in place
    // ---- forward substitution (u into the key tile's bytes), then U~ = e^{G_C - G_s} u_s
    //      as three bf16 tiles (row tid, K = token)
    float *sUf = reinterpret_cast<float *>(sK);                     // [C][128]
    {
        float unused[16];
        blocked_solve(C, tid, lane_base, At, CP, nullptr, sV, sUf, sBeta, sGam, unused);
    }
    __syncthreads();                                                // value rows fully read
#pragma unroll 1
    for (int c8 = 0; c8 < CP / 8; ++c8) {
        __nv_bfloat16 hh[8], mm[8], ll[8];
        const float4 f0 = *reinterpret_cast<const float4 *>(sFold + c8 * 8);
        const float4 f1 = *reinterpret_cast<const float4 *>(sFold + c8 * 8 + 4);
        const float fs[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = c8 * 8 + j;
            const float ut = t < C ? sUf[static_cast<size_t>(t) * 128 + tid] : 0.f;
            split3(fs[j] * ut, hh[j], mm[j], ll[j]);
        }
        const uint32_t off = sw128(tid, c8);
        *reinterpret_cast<uint4 *>(sU + off) =
            make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
        *reinterpret_cast<uint4 *>(sU + 16384 + off) =
            make_uint4(pack2(mm[0], mm[1]), pack2(mm[2], mm[3]), pack2(mm[4], mm[5]), pack2(mm[6], mm[7]));
        *reinterpret_cast<uint4 *>(sU + 32768 + off) =
            make_uint4(pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idF = idesc_mn(1, 128, 128);
        const uint32_t u0 = saddr(sU), kt0 = saddr(sKt);
        for (int sp = 0; sp < 3; ++sp)
            for (int ks = 0; ks < CP / 16; ++ks)
                mma_bf16(tmem, desc_sw128(u0 + sp * 16384 + ks * 32), desc_sw128(kt0 + ks * 32), idF,
                         (sp | ks) != 0);
        mma_commit(&bar[1]);
    }
    ok = mbar_wait(&bar[1], 1);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            mbar_wait(&bar[1], 1);
            atomicOr(a.status, kStatusTimeout);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    tc_fence_after();
    // ---- S_C = gamma_C S0 + D, written over the S0 tile, then one TMA store
    {
        const float gC = sGam[C - 1];
        const int r = tid;
#pragma unroll 2
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float d[16];
            tmem_ld16(lane_base + c0, d);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int col = c0 + 4 * q;                          // 4 fp32 = one 16-byte chunk
                float4 *p = reinterpret_cast<float4 *>(sS + (col >> 5) * 16384 + sw128(r, (col & 31) >> 2));
                float4 x = *p;
                x.x = fmaf(gC, x.x, d[4 * q]);
                x.y = fmaf(gC, x.y, d[4 * q + 1]);
                x.z = fmaf(gC, x.z, d[4 * q + 2]);
                x.w = fmaf(gC, x.w, d[4 * q + 3]);
                *p = x;
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) tma_store_2d(&tm_state, kb * 32, y, sS + kb * 16384);
        tma_store_commit_and_wait();
    }
    __syncthreads();                                                // tiles are reused by the next item
        }
        __syncthreads();                                            // the list is rebuilt
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Fold (flush) through the inverse of the token system.
//
// For the L buffered tokens of one (sequence, head), with D_s = e^{G_{L-1}-G_s} and
// Tinv = (I + A)^{-1}, the checkpoint after the buffer is
//   S_L = gamma_{L-1} S0 + sum_s D_s u_s k_s^T,  u = Tinv r,  r_s = beta_s (v_s - gamma_s S0 k_s),
// and exchanging the sums gives S_L = gamma_{L-1} S0 + R E with the columns r_s in
// R (d_v x L) and E[s'] = sum_s Tinv[s][s'] D_s k_s (L x d_k).  E depends on the tokens
// only, so the triangular work happens on an L x L matrix, not per state row:
//   1. [K] K^T on the tensor cores (bf16 rows as loaded), A in shared memory;
//   2. Tinv by blocks of 16: the diagonal blocks by forward substitution (a thread
//      per column), the blocks below by T_ij = -T_ii sum_k A_ik T_kj, one block
//      diagonal at a time;
//   3. E^T = K^T F^T with F[s'][s] = D_s Tinv[s][s'] split into two bf16 terms, the
//      keys read as an MN-major operand;
//   4. with the checkpoint (TMA from L2, quarters of 32 columns through two 16 KB
//      buffers): S0 K^T in tf32, R in registers, R and E^T each as two bf16 terms,
//      and one M = 128, N = 128 contraction (hi.hi + hi.lo + lo.hi, relative error
//      about 2^-16, far below that of the tf32 S0 K^T).
// Persistent: the CTAs list the sequences that flush (len >= threshold, or len > 0
// when forced) in the same order and take (sequence, head) items with a grid stride.
//
// Shared-memory plan (bytes from the 1024-aligned base), Lp = CMAX:
//   [0, 2 SUBK)            key rows, bf16, 2 sub-tiles of CMAX rows x 128 B
//   [OFF_AT, +Lp^2 4)      A^T, fp32 (row s holds column s of A)
//   [OFF_TI, +Lp^2 4)      Tinv, fp32 row-major
//   [0, 32K)               after E^T is formed: E^T as two bf16 tiles [128][64]
//   [OFF_V, +2 SUBV)       value rows, bf16
//   [OFF_KF, +4 KFSUB)     key rows, fp32, 4 sub-tiles of CMAX rows x 128 B (S0 K^T)
//   [OFF_Q, +32K)          F as two bf16 tiles [CMAX][64] and the block scratch; then
//                          the two checkpoint buffers; then R as two bf16 tiles [128][64]
//   [0, 64K)               after the fold contraction: the new state, for the TMA store
//   [OFF_SC, ...)          mbarriers, TMEM slot, flags, G (hi, lo), beta, gamma, D, list
template <int CMAX> struct FoldPlan {
    static constexpr int SUBK = CMAX * 128;
    static constexpr int OFF_AT = 2 * SUBK;
    static constexpr int OFF_TI = OFF_AT + CMAX * CMAX * 4;
    static constexpr int OFF_V = 32768 > OFF_TI + CMAX * CMAX * 4 ? 32768 : ((OFF_TI + CMAX * CMAX * 4 + 1023) & ~1023);
    static constexpr int SUBV = CMAX * 128;
    static constexpr int OFF_KF = OFF_V + 2 * SUBV;
    static constexpr int KFSUB = CMAX * 128;
    static constexpr int OFF_Q = OFF_KF + 4 * KFSUB;
    static constexpr int OFF_Y = OFF_Q + 2 * CMAX * 128;      // Tinv block scratch (phase A)
    static constexpr int OFF_SC = OFF_Q + 32768;
    static constexpr int LIST = 512;
    static constexpr int BYTES = OFF_SC + 128 + 20 * CMAX + 4 * LIST + 256;
    static_assert(CMAX == 48 || CMAX == 64, "token blocks");
    static_assert(SUBK + 16384 <= OFF_SC, "M = 128 operand reads stay inside the allocation");
    static_assert(OFF_Y + 3 * 1024 <= OFF_SC, "block scratch");
    static_assert(OFF_V >= 32768 && OFF_V + 2 * SUBV + 4 * KFSUB <= OFF_Q, "E^T tiles below the values");
    static_assert(OFF_SC >= 65536, "staging of the new state");
    static_assert((OFF_V % 1024) == 0 && (OFF_KF % 1024) == 0 && (OFF_Q % 1024) == 0 && (SUBK % 1024) == 0 &&
                  (KFSUB % 1024) == 0, "swizzle atoms");
};

template <int CMAX, bool DRAFT>
__global__ void __launch_bounds__(kThreads, 2)
fold_eq_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    using P = FoldPlan<CMAX>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, cap = a.cap;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (saddr(smem_raw) & 1023u) {
        if (tid == 0) atomicOr(a.status, kStatusTimeout);
        return;
    }
    uint8_t *sK = smem_raw;
    float *sAt = reinterpret_cast<float *>(smem_raw + P::OFF_AT);
    float *sTi = reinterpret_cast<float *>(smem_raw + P::OFF_TI);
    uint8_t *sEt = smem_raw;                                      // 2 x 16 KB
    uint8_t *sV = smem_raw + P::OFF_V;
    uint8_t *sKf = smem_raw + P::OFF_KF;
    uint8_t *sF = smem_raw + P::OFF_Q;                            // 2 x CMAX x 128 B
    float *sY = reinterpret_cast<float *>(smem_raw + P::OFF_Y);   // [3][16][16]
    uint8_t *sBuf = smem_raw + P::OFF_Q;                          // 2 x 16 KB
    uint8_t *sR = smem_raw + P::OFF_Q;                            // 2 x 16 KB
    uint8_t *sNew = smem_raw;                                     // 64 KB
    uint8_t *sm = smem_raw + P::OFF_SC;
    // 0: K.K; 1: E^T; 2, 3: checkpoint buffers; 4..7: S0 K^T quarters; 8: fold; 9: draft
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 80);
    int *flag = reinterpret_cast<int *>(sm + 84);
    int *n_list = reinterpret_cast<int *>(sm + 88);
    int *warp_cnt = reinterpret_cast<int *>(sm + 96);              // [4]
    float *sGh = reinterpret_cast<float *>(sm + 128);
    float *sGl = sGh + CMAX;
    float *sBeta = sGl + CMAX;
    float *sGam = sBeta + CMAX;
    float *sD = sGam + CMAX;
    int *list = reinterpret_cast<int *>(sD + CMAX);
    float *dGh = reinterpret_cast<float *>(list + P::LIST);      // draft: G (hi, lo), beta, gamma
    float *dGl = dGh + 16;
    float *dBeta = dGl + 16;
    float *dGam = dBeta + 16;
    constexpr uint32_t COL_KK = 0, COL_E = 64, COL_P = 0, COL_F = 128;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 10; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    pdl_wait();
    pdl_release();
    const uint32_t k0 = saddr(sK), f0 = saddr(sF), kf0 = saddr(sKf), buf0 = saddr(sBuf), r0 = saddr(sR),
                   e0 = saddr(sEt);

    uint32_t it = 0;                                              // items done by this CTA
    bool alive = true;
    for (int b0 = 0; b0 < a.B && alive; b0 += P::LIST) {
        // the list must be identical in every CTA: compact in sequence order with
        // ballots and a prefix over the four warps (no atomics)
        if (tid == 0) *n_list = 0;
        __syncthreads();
        const int bend = min(b0 + P::LIST, a.B);
        for (int g0 = b0; g0 < bend; g0 += kThreads) {
            const int bb = g0 + tid;
            bool f = false;
            if (bb < bend) {
                const int sl = a.state_idx ? a.state_idx[bb] : bb;
                if (sl >= 0 && sl < a.n_slot) {                     // others: reported by the length kernel
                    const int ln = a.buf_len[sl];
                    f = ln >= 0 && ln <= cap && (ln >= a.threshold || (a.force && ln > 0));
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, f);
            if (lane == 0) warp_cnt[warp] = __popc(m);
            __syncthreads();
            int base = *n_list;
            for (int w2 = 0; w2 < warp; ++w2) base += warp_cnt[w2];
            if (f) list[base + __popc(m & ((1u << lane) - 1u))] = bb;
            __syncthreads();
            if (tid == 0) *n_list += warp_cnt[0] + warp_cnt[1] + warp_cnt[2] + warp_cnt[3];
            __syncthreads();
        }
        const int n_items = *n_list * H;
        for (int w = blockIdx.x; w < n_items && alive; w += gridDim.x, ++it) {
            const uint32_t ph = it & 1u;
            const int b = list[w / H], h = w % H;
            const int slot = a.state_idx ? a.state_idx[b] : b;
            const int L = a.buf_len[slot];
            const int Lp = round16(L);
            const int nb = Lp >> 4;
            const size_t unit = static_cast<size_t>(slot) * H + h;
            const int ytile = static_cast<int>(unit) * 128;
            if (tid == 0) {
                *flag = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) prefetch_tile_l2(&tm_state, q * 32, ytile);
            }
            // ---- token rows: keys (bf16 tile, fp32 tile), values (bf16 tile), gates
            const __nv_bfloat16 *bk = reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
            const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
            constexpr int NV = CMAX * 16 / kThreads;
            uint4 raw[NV], vload[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                raw[i] = make_uint4(0u, 0u, 0u, 0u);
                vload[i] = make_uint4(0u, 0u, 0u, 0u);
                if (r < L) {
                    raw[i] = __ldg(reinterpret_cast<const uint4 *>(bk + static_cast<size_t>(r) * 128) + c);
                    vload[i] = __ldg(reinterpret_cast<const uint4 *>(bv + static_cast<size_t>(r) * 128) + c);
                }
            }
            float gq[2] = {0.f, 0.f}, bq[2] = {0.f, 0.f};
            if (warp == 0) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int t = lane + 32 * i;
                    if (t < L) {
                        gq[i] = a.buf_g[unit * cap + t];
                        bq[i] = a.buf_beta[unit * cap + t];
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                *reinterpret_cast<uint4 *>(sK + (c >> 3) * P::SUBK + sw128(r, c & 7)) = raw[i];
                *reinterpret_cast<uint4 *>(sV + (c >> 3) * P::SUBV + sw128(r, c & 7)) = vload[i];
                float fl[8];
                bf16x8_to_f32(raw[i], fl);
                uint8_t *tile = sKf + (c >> 2) * P::KFSUB;
                const int ch = (c & 3) * 2;
                *reinterpret_cast<float4 *>(tile + sw128(r, ch)) = make_float4(fl[0], fl[1], fl[2], fl[3]);
                *reinterpret_cast<float4 *>(tile + sw128(r, ch + 1)) = make_float4(fl[4], fl[5], fl[6], fl[7]);
            }
            if (warp == 0) {                                      // compensated scan of g
                float hi[2], lo[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    hi[i] = gq[i];
                    lo[i] = 0.f;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float h2 = __shfl_up_sync(0xffffffffu, hi[i], off);
                        const float l2 = __shfl_up_sync(0xffffffffu, lo[i], off);
                        if (lane >= off) {
                            const float s1 = hi[i] + h2, bp = s1 - hi[i];
                            lo[i] += l2 + ((hi[i] - (s1 - bp)) + (h2 - bp));
                            hi[i] = s1;
                        }
                    }
                }
                const float chh = __shfl_sync(0xffffffffu, hi[0], 31), cll = __shfl_sync(0xffffffffu, lo[0], 31);
                {
                    const float s1 = hi[1] + chh, bp = s1 - hi[1];
                    lo[1] += cll + ((hi[1] - (s1 - bp)) + (chh - bp));
                    hi[1] = s1;
                }
                // G_{L-1} (hi, lo) from the lane that holds it
                const int src = (L - 1) & 31;
                const float gLh = __shfl_sync(0xffffffffu, (L - 1) >= 32 ? hi[1] : hi[0], src);
                const float gLl = __shfl_sync(0xffffffffu, (L - 1) >= 32 ? lo[1] : lo[0], src);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int t = lane + 32 * i;
                    if (t < CMAX) {
                        const bool live = t < L;
                        sGh[t] = live ? hi[i] : 0.f;
                        sGl[t] = live ? lo[i] : 0.f;
                        sGam[t] = live ? __expf(hi[i] + lo[i]) : 0.f;
                        sBeta[t] = live ? bq[i] : 0.f;
                        sD[t] = live ? __expf((gLh - hi[i]) + (gLl - lo[i])) : 0.f;
                    }
                }
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {                                       // K K^T
                tc_fence_after();
                const uint32_t idK = idesc_mn(1, 128, Lp);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = desc_sw128(k0 + (ks >> 2) * P::SUBK + (ks & 3) * 32);
                    mma_bf16(tmem + COL_KK, d, d, idK, ks > 0);
                }
                mma_commit(&bar[0]);
            }
            bool ok = mbar_wait(&bar[0], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) { mbar_wait(&bar[0], ph); atomicOr(a.status, kStatusTimeout); }
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- A^T: thread t writes column t of A (row t of A^T): A[t][s] for s < t
            if (warp * 32 < CMAX) {                               // warp-uniform: collective loads
                const int t = tid;
                const float gh = t < L ? sGh[t] : 0.f, gl = t < L ? sGl[t] : 0.f, bt = t < L ? sBeta[t] : 0.f;
#pragma unroll
                for (int cb = 0; cb < CMAX / 16; ++cb) {
                    const int c0 = cb * 16;
                    float kk[16];
                    if (c0 < Lp) {
                        tmem_ld16(lane_base + COL_KK + c0, kk);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) kk[j] = 0.f;
                    }
                    float gs[16], ls[16], av[16];
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 x = *reinterpret_cast<const float4 *>(sGh + c0 + 4 * j4);
                        const float4 y = *reinterpret_cast<const float4 *>(sGl + c0 + 4 * j4);
                        gs[4 * j4] = x.x; gs[4 * j4 + 1] = x.y; gs[4 * j4 + 2] = x.z; gs[4 * j4 + 3] = x.w;
                        ls[4 * j4] = y.x; ls[4 * j4 + 1] = y.y; ls[4 * j4 + 2] = y.z; ls[4 * j4 + 3] = y.w;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = c0 + j;
                        const float e = __expf((gh - gs[j]) + (gl - ls[j]));
                        av[j] = (s < t && t < L) ? bt * e * kk[j] : 0.f;
                    }
                    if (t < CMAX) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) sAt[(c0 + j) * CMAX + t] = av[j];
                    }
                }
            }
            __syncthreads();
            // ---- Tinv, diagonal blocks: thread j < Lp solves column j of its block
            if (tid < Lp) {
                const int j = tid, kb = j >> 4, c = j & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = i == c ? 1.f : 0.f;
#pragma unroll
                for (int l = 0; l < 15; ++l) {
                    if (l >= c) {
                        const float xl = x[l];
                        const float4 *arow = reinterpret_cast<const float4 *>(sAt + (16 * kb + l) * CMAX + 16 * kb);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 av = arow[q];
                            if (4 * q > l) x[4 * q] = fmaf(-av.x, xl, x[4 * q]);
                            if (4 * q + 1 > l) x[4 * q + 1] = fmaf(-av.y, xl, x[4 * q + 1]);
                            if (4 * q + 2 > l) x[4 * q + 2] = fmaf(-av.z, xl, x[4 * q + 2]);
                            if (4 * q + 3 > l) x[4 * q + 3] = fmaf(-av.w, xl, x[4 * q + 3]);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < CMAX; ++i) {                  // the whole column (zeros off the block)
                    const int ib = i >> 4;
                    sTi[i * CMAX + j] = ib == kb ? x[i & 15] : 0.f;
                }
            }
            __syncthreads();
            // ---- blocks below the diagonal, one block diagonal d at a time:
            //      Y_j = sum_{k=j}^{j+d-1} A_{j+d,k} T_{k,j};  T_{j+d,j} = -T_{j+d,j+d} Y_j
            for (int d = 1; d < nb; ++d) {
                const int nblk = nb - d;
                // a task: block j, row r, columns 4 c4 .. 4 c4 + 3
                for (int e = tid; e < nblk * 64; e += kThreads) {
                    const int j = e >> 6, r = (e >> 2) & 15, c4 = e & 3, i = j + d;
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int k = j; k < i; ++k) {
#pragma unroll
                        for (int l = 0; l < 16; ++l) {
                            const float av = sAt[(16 * k + l) * CMAX + 16 * i + r];
                            const float4 tv = *reinterpret_cast<const float4 *>(sTi + (16 * k + l) * CMAX + 16 * j + 4 * c4);
                            y.x = fmaf(av, tv.x, y.x); y.y = fmaf(av, tv.y, y.y);
                            y.z = fmaf(av, tv.z, y.z); y.w = fmaf(av, tv.w, y.w);
                        }
                    }
                    *reinterpret_cast<float4 *>(sY + (j << 8) + r * 16 + 4 * c4) = y;
                }
                __syncthreads();
                for (int e = tid; e < nblk * 64; e += kThreads) {
                    const int j = e >> 6, r = (e >> 2) & 15, c4 = e & 3, i = j + d;
                    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int l = 0; l < 16; ++l) {
                        const float tv = sTi[(16 * i + r) * CMAX + 16 * i + l];
                        const float4 yv = *reinterpret_cast<const float4 *>(sY + (j << 8) + l * 16 + 4 * c4);
                        t.x = fmaf(tv, yv.x, t.x); t.y = fmaf(tv, yv.y, t.y);
                        t.z = fmaf(tv, yv.z, t.z); t.w = fmaf(tv, yv.w, t.w);
                    }
                    *reinterpret_cast<float4 *>(sTi + (16 * i + r) * CMAX + 16 * j + 4 * c4) =
                        make_float4(-t.x, -t.y, -t.z, -t.w);
                }
                __syncthreads();
            }
            // ---- F[s'][s] = D_s Tinv[s][s'] as two bf16 K-major tiles [Lp][64]
            for (int e = tid; e < Lp * 64 / 8; e += kThreads) {
                const int sp = e >> 3, c8 = e & 7;                // row s', 8 columns s = 8 c8 ..
                __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int s = c8 * 8 + j;
                    const float v = s < CMAX ? sD[s] * sTi[s * CMAX + sp] : 0.f;
                    split2(v, hh[j], ll[j]);
                }
                const uint32_t off = sw128(sp, c8);
                *reinterpret_cast<uint4 *>(sF + off) =
                    make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                *reinterpret_cast<uint4 *>(sF + CMAX * 128 + off) =
                    make_uint4(pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {                                       // E^T = K^T F^T (keys MN-major)
                tc_fence_after();
                const uint32_t idE = idesc_mn(1, 128, Lp) | kIdescMnMajorA;
                for (int ks = 0; ks < nb; ++ks) {
                    const uint64_t ak = desc_mn_sw128(k0 + ks * 2048, P::SUBK);
                    mma_bf16(tmem + COL_E, ak, desc_sw128(f0 + ks * 32), idE, ks > 0);
                    mma_bf16(tmem + COL_E, ak, desc_sw128(f0 + CMAX * 128 + ks * 32), idE, 1);
                }
                mma_commit(&bar[1]);
            }
            ok = mbar_wait(&bar[1], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) { mbar_wait(&bar[1], ph); atomicOr(a.status, kStatusTimeout); }
                alive = false;
                break;
            }
            tc_fence_after();
            // the checkpoint quarters 0, 1 come in from L2 (F is no longer read)
            if (tid == 0) {
                fence_proxy_async();
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    mbar_expect_tx(&bar[2 + q], 16384);
                    tma_load_2d(sBuf + q * 16384, &tm_state, q * 32, ytile, &bar[2 + q]);
                }
            }
            // ---- E^T row d_k = tid as two bf16 terms, K-major [128][64] tiles
#pragma unroll
            for (int cb = 0; cb < CMAX / 16; ++cb) {
                if (cb < nb) {
                    float ev[16];
                    tmem_ld16(lane_base + COL_E + cb * 16, ev);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) split2(ev[8 * hf + j], hh[j], ll[j]);
                        const uint32_t off = sw128(tid, 2 * cb + hf);
                        *reinterpret_cast<uint4 *>(sEt + off) = make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]),
                                                                           pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                        *reinterpret_cast<uint4 *>(sEt + 16384 + off) = make_uint4(
                            pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
                    }
                }
            }
            // ---- S0 K^T, quarter by quarter (thread 0), into the K K^T columns
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idP = idesc_mn(2, 128, Lp);
                int loads[2] = {1, 1}, mmas = 0;
                bool good = true;
                for (int q = 0; q < 4; ++q) {
                    const int bi = q & 1;
                    if (!mbar_wait(&bar[2 + bi], q >> 1)) { good = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_tf32(tmem + COL_P, desc_sw128(buf0 + bi * 16384 + ks * 32),
                                 desc_sw128(kf0 + q * P::KFSUB + ks * 32), idP, (q | ks) != 0);
                    mma_commit(&bar[4 + q]);
                    mmas = q + 1;
                    if (q < 2) {
                        if (!mbar_wait(&bar[4 + q], ph)) { good = false; break; }
                        mbar_expect_tx(&bar[2 + bi], 16384);
                        tma_load_2d(sBuf + bi * 16384, &tm_state, (q + 2) * 32, ytile, &bar[2 + bi]);
                        ++loads[bi];
                    }
                }
                if (!good) {
                    for (int q = 0; q < mmas; ++q) mbar_wait(&bar[4 + q], ph);
                    for (int i = 0; i < 2; ++i) mbar_wait(&bar[2 + i], (loads[i] - 1) & 1);
                    *flag = 1;
                }
            }
            __syncthreads();
            ok = *flag == 0;
            if (ok) ok = mbar_wait(&bar[7], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    if (*flag == 0) mbar_wait(&bar[7], ph);
                    atomicOr(a.status, kStatusTimeout);
                }
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- R row d_v = tid: r_s = beta_s (v_s - gamma_s (S0 k_s)), two bf16 terms
            {
                const uint8_t *vcol = sV + (tid >> 6) * P::SUBV + (tid & 7) * 2;
                const int vch = (tid & 63) >> 3;
#pragma unroll
                for (int cb = 0; cb < CMAX / 16; ++cb) {
                    if (cb < nb) {
                        float pk[16];
                        tmem_ld16(lane_base + COL_P + cb * 16, pk);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int s = cb * 16 + 8 * hf + j;
                                const float v = __bfloat162float(
                                    *reinterpret_cast<const __nv_bfloat16 *>(vcol + sw128(s, vch)));
                                split2(sBeta[s] * (v - sGam[s] * pk[8 * hf + j]), hh[j], ll[j]);
                            }
                            const uint32_t off = sw128(tid, 2 * cb + hf);
                            *reinterpret_cast<uint4 *>(sR + off) = make_uint4(
                                pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                            *reinterpret_cast<uint4 *>(sR + 16384 + off) = make_uint4(
                                pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
                        }
                    }
                }
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {                                       // D = R E: hi.hi + hi.lo + lo.hi
                tc_fence_after();
                const uint32_t idF = idesc_mn(1, 128, 128);
                for (int ks = 0; ks < nb; ++ks) {
                    const uint64_t rh = desc_sw128(r0 + ks * 32), rl = desc_sw128(r0 + 16384 + ks * 32);
                    const uint64_t eh = desc_sw128(e0 + ks * 32), el = desc_sw128(e0 + 16384 + ks * 32);
                    mma_bf16(tmem + COL_F, rh, eh, idF, ks > 0);
                    mma_bf16(tmem + COL_F, rh, el, idF, 1);
                    mma_bf16(tmem + COL_F, rl, eh, idF, 1);
                }
                mma_commit(&bar[8]);
            }
            // rows 32 warp .. 32 warp + 31 of S0 (L2), 512 contiguous bytes per warp load,
            // while the contraction runs
            float4 *srow = reinterpret_cast<float4 *>(a.state_out + (unit * 128 + 32 * warp) * 128) + lane;
            float4 x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = srow[i * 32];
            ok = mbar_wait(&bar[8], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) { mbar_wait(&bar[8], ph); atomicOr(a.status, kStatusTimeout); }
                alive = false;
                break;
            }
            tc_fence_after();
            // the draft rows ([K_d; Q_d] as 32 rows, V_d) and gates, for the verify below
            uint4 dkq[4], dvv[2];
            float dgq = 0.f, dbq = 0.f;
            const size_t drow0 = (static_cast<size_t>(b) * a.T * H + h) * 128;
            if constexpr (DRAFT) {
                const size_t dstride = static_cast<size_t>(H) * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    const int t = r & 15;
                    dkq[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (t < a.T)
                        dkq[i] = __ldg(reinterpret_cast<const uint4 *>(
                                           reinterpret_cast<const __nv_bfloat16 *>(r < 16 ? a.k : a.q) + drow0 +
                                           static_cast<size_t>(t) * dstride) + c);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    dvv[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (r < a.T)
                        dvv[i] = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.v) +
                                                                       drow0 + static_cast<size_t>(r) * dstride) + c);
                }
                if (warp == 0 && lane < a.T) {
                    const size_t gi = (static_cast<size_t>(b) * a.T + lane) * H + h;
                    dgq = a.g[gi];
                    dbq = a.beta[gi];
                }
            }
            // ---- D row tid into shared memory (swizzled rows), then S_L = gamma_{L-1} S0 + D
            //      row by row with coalesced loads and stores
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 16) {
                float dd[16];
                tmem_ld16(lane_base + COL_F + c0, dd);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = c0 + 4 * q;
                    *reinterpret_cast<float4 *>(sNew + (col >> 5) * 16384 + sw128(tid, (col & 31) >> 2)) =
                        make_float4(dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
                }
            }
            __syncwarp();                                         // a warp reads back only its own rows
            {
                const float gL = sGam[L - 1];
                const uint8_t *dsub = sNew + (lane >> 3) * 16384;
                float4 x2[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x2[i] = srow[(16 + i) * 32];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int row = 16 * hf + i;
                        const float4 dv4 = *reinterpret_cast<const float4 *>(dsub + sw128(32 * warp + row, lane & 7));
                        float4 y = hf ? x2[i] : x[i];
                        y.x = fmaf(gL, y.x, dv4.x);
                        y.y = fmaf(gL, y.y, dv4.y);
                        y.z = fmaf(gL, y.z, dv4.z);
                        y.w = fmaf(gL, y.w, dv4.w);
                        srow[row * 32] = y;
                        if constexpr (DRAFT)                     // S_L stays as the operand of the draft
                            *reinterpret_cast<float4 *>(const_cast<uint8_t *>(dsub) + sw128(32 * warp + row, lane & 7)) = y;
                    }
                }
            }
            if constexpr (DRAFT) {
                // ---- the draft, verified from the new state S_L (buffer now empty): with G'
                //      the running sum over the draft alone, u' from the 16-token system and
                //      o_t2 = scale (gamma'_t2 S_L q_t2 + sum_{s<=t2} e^{G'_t2-G'_s} (q_t2.k_s) u'_s);
                //      the draft is staged at buffer slot 0
                const int T = a.T;
                uint8_t *sDq = sR;                                // [K_d; Q_d] fp32, 4 sub-tiles of 32 x 128 B
                __nv_bfloat16 *sVd = reinterpret_cast<__nv_bfloat16 *>(sR + 16384);   // [16][128]
                float *sAtd = reinterpret_cast<float *>(sR + 20480);                  // A'^T [16][16]
                float *sMtd = sAtd + 256;                                             // M'^T [16][16]
                float *sUd = reinterpret_cast<float *>(sR + 22528);                   // u' [16][128]
                __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
                __nv_bfloat16 *wv = reinterpret_cast<__nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    float fl[8];
                    bf16x8_to_f32(dkq[i], fl);
                    uint8_t *tile = sDq + (c >> 2) * 4096;
                    const int ch = (c & 3) * 2;
                    *reinterpret_cast<float4 *>(tile + sw128(r, ch)) = make_float4(fl[0], fl[1], fl[2], fl[3]);
                    *reinterpret_cast<float4 *>(tile + sw128(r, ch + 1)) = make_float4(fl[4], fl[5], fl[6], fl[7]);
                    if (r < T) reinterpret_cast<uint4 *>(wk + static_cast<size_t>(r) * 128)[c] = dkq[i];
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    reinterpret_cast<uint4 *>(sVd + static_cast<size_t>(r) * 128)[c] = dvv[i];
                    if (r < T) reinterpret_cast<uint4 *>(wv + static_cast<size_t>(r) * 128)[c] = dvv[i];
                }
                if (warp == 0) {                                  // compensated scan over the draft
                    float hi = dgq, lo = 0.f;
#pragma unroll
                    for (int off = 1; off < 16; off <<= 1) {
                        const float h2 = __shfl_up_sync(0xffffffffu, hi, off);
                        const float l2 = __shfl_up_sync(0xffffffffu, lo, off);
                        if (lane >= off) {
                            const float s1 = hi + h2, bp = s1 - hi;
                            lo += l2 + ((hi - (s1 - bp)) + (h2 - bp));
                            hi = s1;
                        }
                    }
                    if (lane < 16) {
                        const bool live = lane < T;
                        dGh[lane] = live ? hi : 0.f;
                        dGl[lane] = live ? lo : 0.f;
                        dGam[lane] = live ? __expf(hi + lo) : 0.f;
                        dBeta[lane] = live ? dbq : 0.f;
                        if (live) {
                            a.buf_g[unit * cap + lane] = dgq;
                            a.buf_beta[unit * cap + lane] = dbq;
                        }
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncthreads();
                const uint32_t dq0 = saddr(sDq), sn0 = saddr(sNew);
                if (tid == 0) {                                   // [K_d;Q_d] K_d^T and S_L [K_d;Q_d]^T
                    tc_fence_after();
                    const uint32_t idK = idesc_mn(2, 128, 16), idP = idesc_mn(2, 128, 32);
#pragma unroll
                    for (int ks = 0; ks < 16; ++ks) {
                        const uint64_t dd = desc_sw128(dq0 + (ks >> 2) * 4096 + (ks & 3) * 32);
                        mma_tf32(tmem + 0, dd, dd, idK, ks > 0);
                        mma_tf32(tmem + 16, desc_sw128(sn0 + (ks >> 2) * 16384 + (ks & 3) * 32), dd, idP, ks > 0);
                    }
                    mma_commit(&bar[9]);
                }
                ok = mbar_wait(&bar[9], ph);
                if (__syncthreads_or(!ok)) {
                    if (tid == 0) { mbar_wait(&bar[9], ph); atomicOr(a.status, kStatusTimeout); }
                    alive = false;
                    break;
                }
                tc_fence_after();
                if (warp == 0) {                                  // lanes 0..15: A' rows, 16..31: M' rows
                    float kq[16];
                    tmem_ld16(lane_base + 0, kq);
                    const bool is_q = lane >= 16;
                    const int t = lane & 15;
                    const float gh = dGh[t], gl = dGl[t], scl = is_q ? 1.f : dBeta[t];
                    const int lim = t >= T ? 0 : is_q ? t + 1 : t;
                    float *dst = (is_q ? sMtd : sAtd) + t;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float e = __expf((gh - dGh[j]) + (gl - dGl[j]));
                        dst[j * 16] = j < lim ? scl * e * kq[j] : 0.f;
                    }
                }
                __syncthreads();
                float od[16];
                blocked_solve(T, tid, lane_base + 16, sAtd, 16, sMtd, sVd, sUd, dBeta, dGam, od);
                float pq[16];
                tmem_ld16(lane_base + 32, pq);
#pragma unroll
                for (int t2 = 0; t2 < 16; ++t2)
                    if (t2 < T)
                        a.out[((static_cast<size_t>(b) * T + t2) * H + h) * 128 + tid] =
                            a.scale * (dGam[t2] * pq[t2] + od[t2]);
            }
            tc_fence_before();
            __syncthreads();                                      // the tiles are reused by the next item
        }
        __syncthreads();                                          // the list is rebuilt
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// The checkpoint as a 2-D fp32 tensor [n_slot*H*128 rows, 128 cols]; boxes of
// 32 columns (128 bytes) x 128 rows, 128-byte swizzle.
bool state_map(CUtensorMap *m, const float *state, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {128 * sizeof(float)};
    cuuint32_t box[2] = {32, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(state), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of one launch that can be resident at once (the prefetch distance).
int resident_ctas(const void *kern, int smem) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
        return 0;
    return sms * per_sm;
}

template <int CMAX>
int launch_eq(const gdn_replay_dims *d, const ReplayArgs &a, const CUtensorMap &m, cudaStream_t s) {
    constexpr int smem = EqPlan<CMAX>::BYTES;
    auto kern = verify_eq_kernel<CMAX>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    return launch_pdl(kern, dim3(d->H, d->B), dim3(kThreads), smem, s, m, a) == cudaSuccess ? GDN_OK
                                                                                       : GDN_ERR_LAUNCH;
}

template <int CMAX, bool FOLD>
int launch_verify(const gdn_replay_dims *d, const ReplayArgs &a0, const CUtensorMap &m, cudaStream_t s) {
    const int smem = verify_smem_bytes(FOLD ? d->cap + d->T : d->cap, d->T);
    auto kern = verify_tc_kernel<CMAX, FOLD>;
    static int stride = -1;                                       // per instantiation, per process
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    if (stride < 0) stride = resident_ctas(reinterpret_cast<const void *>(kern), smem);
    ReplayArgs a = a0;
    a.prefetch_stride = stride;
    return launch_pdl(kern, dim3(d->H, d->B), dim3(kThreads), smem, s, m, a) == cudaSuccess ? GDN_OK
                                                                                       : GDN_ERR_LAUNCH;
}

template <bool DRAFT>
int launch_fold(const gdn_replay_dims *d, const ReplayArgs &a, const CUtensorMap &m, cudaStream_t s) {
    const bool small = d->cap <= 48;
    const int smem = small ? FoldPlan<48>::BYTES : FoldPlan<64>::BYTES;
    auto kern = small ? fold_eq_kernel<48, DRAFT> : fold_eq_kernel<64, DRAFT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    int ctas = resident_ctas(reinterpret_cast<const void *>(kern), smem);
    if (ctas <= 0) return GDN_ERR_LAUNCH;
    ctas = ctas < d->B * d->H ? ctas : d->B * d->H;
    return launch_pdl(kern, dim3(ctas), dim3(kThreads), smem, s, m, a) == cudaSuccess ? GDN_OK
                                                                                 : GDN_ERR_LAUNCH;
}

}  // namespace

int tc_verify(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s, bool fold) {
    if (d->dk != 128 || d->dv != 128 || d->in_dtype != GDN_DTYPE_BF16) return 1;
    const int cmax = fold ? d->cap + d->T : d->cap;               // tokens one unit may replay
    if (cmax > 64 || d->T > 16) return 1;                         // register arrays hold 64 tokens
    if (verify_smem_bytes(cmax, d->T) > 227 * 1024) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_in, d->n_slot * d->H * 128)) return 1;
    if (!fold) return cmax <= 48 ? launch_eq<48>(d, a, m, s) : launch_eq<64>(d, a, m, s);
    return cmax <= 48 ? launch_verify<48, true>(d, a, m, s) : launch_verify<64, true>(d, a, m, s);
}


int tc_flush(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    if (d->dk != 128 || d->dv != 128 || d->in_dtype != GDN_DTYPE_BF16) return 1;
    if (d->cap > 64) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_out, d->n_slot * d->H * 128)) return 1;
    return launch_fold<false>(d, a, m, s);
}

int tc_verify_fold_split(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    if (d->dk != 128 || d->dv != 128 || d->in_dtype != GDN_DTYPE_BF16) return 1;
    if (d->cap > 64 || d->T > 16) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_out, d->n_slot * d->H * 128)) return 1;
    ReplayArgs af = a;                                            // fold the full buffers, verify the draft
    af.force = 0;
    const int rc = launch_fold<true>(d, af, m, s);
    if (rc) return rc;
    ReplayArgs an = a;                                            // the rest, beside the fold launch
    an.fold_class = 1;
    return d->cap <= 48 ? launch_eq<48>(d, an, m, s) : launch_eq<64>(d, an, m, s);
}

}  // namespace gdn
