// gdn_replay_tc.cu -- tensor-core (tcgen05) verify / fold kernels of libgdnreplay
// for sm_103a, for d_k = d_v = 128, bf16 inputs, T <= 16 and buffers of at most 64
// tokens.
//
// Chunked form.  For one (sequence, head) replaying C tokens (the committed
// buffer, then the draft block) from the checkpoint S0, with G_t the running
// sum of the log-decays g and gamma_t = e^{G_t}, the gated delta rule
// ("Gated Delta Networks", ICLR 2025) unrolls into the chunkwise (UT) form of
// "Parallelizing Linear Transformers with the Delta Rule over Sequence
// Length" (NeurIPS 2024):
//   u = (I + A)^{-1} r,  A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s) (s < t),
//   r_t = beta_t (v_t - gamma_t S0 k_t),
//   o_t = scale (gamma_t S0 q_t + sum_{s<=t} e^{G_t-G_s} (q_t.k_s) u_s),
//   S_C = gamma_{C-1} S0 + sum_s e^{G_{C-1}-G_s} u_s k_s^T.
// Both kernels move the triangular algebra onto the C x C token system, which does
// not involve the checkpoint, so S0 enters only dense d_v x d_k contractions:
//   verify_eq_kernel  o = scale (S0 qe + ve) with W = M (I + A)^{-1} (effective
//                     queries, one N = 16 contraction with S0);
//   fold_eq_kernel    S_L = gamma S0 + (V^T + R') E' with E' = diag(beta) Tinv^T D K
//                     (a blocked inverse of the L x L system), then, in the fused
//                     step, the draft verified from S_L.
// Only differences G_t - G_s <= 0 are exponentiated (G kept as a compensated pair).
//
// Data movement: checkpoint tiles arrive by TMA with 128-byte swizzle (the K-major
// layout tcgen05 reads); key and value rows are staged as bf16 swizzled tiles and
// read by the tensor cores either K-major or MN-major (so no transposes are built).
// Accumulators live in TMEM and are read back with tcgen05.ld.  Every wait is
// bounded: on expiry the unit is skipped, a status bit is set, and the kernel still
// waits (bounded) for its own copies and MMAs before freeing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "replay_common.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 128;               // one thread per state row / TMEM lane
constexpr int kTmemCols = 256;
// Registers of a fold thread: one fold CTA (and its 256 TMEM columns) leaves room on
// its SM for three verify CTAs (3 x 128 x 96 + 128 x 224 = 65536).
constexpr int kFoldRegs = 224;

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
// rows and one lane per token column modulo 32; qe and ve are bf16 contractions of the
// key and value rows (read as MN-major operands, no transpose) with W beta gamma
// and W beta split into two bf16 terms each (relative error 2^-16).
// The checkpoint is prefetched into L2 at the start and streamed through two
// 16 KB buffers in quarters of 32 columns once the token work is done.
//
// Shared-memory plan (bytes from the 1024-aligned base), NPA = round16(CMAX + 16):
//   [0, 2 SUBV)          value rows, bf16, 2 sub-tiles (d_k halves) of CMAX rows x 128 B
//   [OFF_K, +2 SUBK)     [K;Q] rows, bf16, 2 sub-tiles of NPA rows x 128 B
//   [OFF_A, +CMAX^2 4)   A, fp32, row-major [CMAX][CMAX]
//   [OFF_M, +16 CMAX 4)  M, fp32, row-major [16][CMAX]
//   [OFF_A, +8K)         after the back substitution: W beta gamma and W beta as 2 + 2
//                        bf16 tiles [16][64]; CMAX = 80: token columns 64..79 in 2 + 2
//                        tiles [16][16] with 32-byte swizzle at [OFF_A + 8K, +2K)
//   [0, 32K)             after the token contractions: two checkpoint quarter buffers
//   [OFF_QE, +8K)        then qe as fp32 [16][128] (4 sub-tiles of 16 rows x 128 B)
//   [OFF_S, ...)         8 mbarriers, TMEM slot, flag, then G (hi, lo), beta, gamma
// An M = 128 operand starting in the [K;Q] tile reads on past its NPA rows; those
// rows only feed accumulator lanes that are never read.  [K;Q] K^T is formed as two
// MMAs: lanes 0..63 get rows 0..63 and the first columns, and, from an operand that
// starts 64 rows before the tile, lanes 64..127 get rows 0..63 and the remaining
// columns, so all four warps build coefficients.
template <int CMAX> struct EqPlan {
    static constexpr int NPL = (CMAX + 31) / 32;              // token columns per lane
    static constexpr bool TAIL = CMAX > 64;                   // K atoms of 64 tokens + 16
    static constexpr int W_BYTES = 8192 + (TAIL ? 2048 : 0);
    static constexpr int NPA = (CMAX + 16 + 15) & ~15;
    static constexpr int SUBK = NPA * 128;
    static constexpr int SUBV = CMAX * 128;
    static constexpr int OFF_K = 2 * SUBV;
    static constexpr int OFF_A = OFF_K + 2 * SUBK;
    static constexpr int OFF_M = OFF_A + CMAX * CMAX * 4;
    static constexpr int OFF_W = OFF_A;                       // over A and M, once they are read
    static constexpr int OFF_QE = 32768;                      // past the two quarter buffers
    static constexpr int A_END = OFF_M + 16 * CMAX * 4;
    static constexpr int OFF_S = ((A_END > OFF_QE + 8192 ? A_END : OFF_QE + 8192) + 127) & ~127;
    static constexpr int BYTES = OFF_S + 128 + 16 * CMAX;
    // TMEM: K.K in [0, CMAX) (then ve, O over it), qe^T in [CMAX, CMAX + 16)
    static constexpr int TMEM_COLS = CMAX + 16 <= 64 ? 64 : 128;
    static constexpr int BLOCKS_PER_SM = CMAX + 16 <= 64 ? 5 : CMAX <= 64 ? 3 : 2;
    static_assert(OFF_W % 1024 == 0 && OFF_W + W_BYTES <= A_END, "W tiles over A and M");
    static_assert(OFF_QE >= 32768 && OFF_QE + 8192 <= OFF_S, "qe tile past the quarter buffers");
    static_assert(OFF_K + SUBK + 16384 <= BYTES, "M = 128 operand reads stay inside the allocation");
    static_assert(OFF_K >= 8192, "an operand may start 64 rows before the [K;Q] tile");
    static_assert(CMAX % 16 == 0 && (CMAX <= 64 || CMAX == 80), "token columns: one 64-token atom, then 16");
    static_assert((SUBK % 1024) == 0 && (OFF_K % 1024) == 0 && (SUBV % 1024) == 0, "swizzle atoms");
};


template <int CMAX>
__global__ void __launch_bounds__(kThreads, EqPlan<CMAX>::BLOCKS_PER_SM)
verify_eq_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    using P = EqPlan<CMAX>;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, H = a.H, cap = a.cap;

    // fold_class 1: the units that do not fold, in a launch that runs beside the fold
    // launch preceding it and must not wait for it (every CTA of that launch has
    // waited for the earlier kernels before letting this one start); CTA (0, 0) waits
    // for it at the end instead, so the next kernel observes both launches complete.
    // It reports the length errors of every sequence (the fold launch skips them).
    const bool split = a.fold_class == 1;
    const bool waiter = split && blockIdx.x == 0 && blockIdx.y == 0;
    // GDN_FLAG_TEST_EXPIRE: take the wait-expiry exit at the first bounded wait, with
    // nothing issued before it
    const bool expire = (a.flags & GDN_FLAG_TEST_EXPIRE) != 0;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (saddr(smem_raw) & 1023u) {           // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) atomicOr(a.status, kStatusTimeout);
        if (waiter) pdl_wait();
        return;
    }
    uint8_t *sV = smem_raw;
    uint8_t *sKQ = smem_raw + P::OFF_K;
    float *sAm = reinterpret_cast<float *>(smem_raw + P::OFF_A);
    float *sMm = reinterpret_cast<float *>(smem_raw + P::OFF_M);
    uint8_t *sW = smem_raw + P::OFF_W;
    uint8_t *sQe = smem_raw + P::OFF_QE;
    uint8_t *sm = smem_raw + P::OFF_S;
    // 0, 1: checkpoint buffers (TMA); 2: K.K; 3: qe, ve; 4..7: checkpoint quarter MMAs
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 64);
    int *flag = reinterpret_cast<int *>(sm + 68);
    float *sGh = reinterpret_cast<float *>(sm + 128);
    float *sGl = sGh + CMAX;
    float *sBeta = sGl + CMAX;
    float *sGam = sBeta + CMAX;
    constexpr int COL_Q = CMAX, COL_V = 0, COL_O = 16;           // TMEM columns (ve, O over K.K)

    if (tid == 0) {                                               // prologue: no global memory
#pragma unroll
        for (int i = 0; i < 8; ++i) mbar_init(&bar[i], 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, P::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (!split) pdl_wait();

    // ---- the draft rows first: their addresses do not depend on the buffer length,
    //      so they are in flight while the slot and the length are read.  Vector i of
    //      a thread is row (tid >> 4) + 8 (i & 1) of the draft keys (i < 2), queries
    //      (i < 4) or values, 16-byte column tid & 15.
    const size_t drow0 = (static_cast<size_t>(b) * T * H + h) * 128;
    const size_t dstride = static_cast<size_t>(H) * 128;
    const __nv_bfloat16 *dk = reinterpret_cast<const __nv_bfloat16 *>(a.k) + drow0;
    const __nv_bfloat16 *dq = reinterpret_cast<const __nv_bfloat16 *>(a.q) + drow0;
    const __nv_bfloat16 *dv = reinterpret_cast<const __nv_bfloat16 *>(a.v) + drow0;
    const int dj = tid >> 4, dc = tid & 15;                       // draft row (+ 8), column vector
    uint4 draft[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        const int j = dj + 8 * (i & 1);
        const __nv_bfloat16 *src = i < 2 ? dk : i < 4 ? dq : dv;
        draft[i] = j < T ? __ldg(reinterpret_cast<const uint4 *>(src + static_cast<size_t>(j) * dstride) + dc)
                         : make_uint4(0u, 0u, 0u, 0u);
    }
    float dg = 0.f, db = 0.f;                                     // warp 0: draft token `lane`
    if (warp == 0 && lane < T) {
        const size_t gi = (static_cast<size_t>(b) * T + lane) * H + h;
        dg = a.g[gi];
        db = a.beta[gi];
    }

    const int slot = a.state_idx ? a.state_idx[b] : b;
    const int len = (slot >= 0 && slot < a.n_slot) ? a.buf_len[slot] : 0;
    const bool other_class = split && len >= a.threshold && len <= cap;   // the fold launch's unit
    int bad = 0;
    if (slot < 0 || slot >= a.n_slot) bad = GDN_STATUS_BAD_SLOT;
    else if (len < 0 || len > cap) bad = GDN_STATUS_BAD_LEN;
    else if (!other_class && len + T > cap) bad = GDN_STATUS_NO_ROOM;
    // launch_dependents comes only before the epilogue: the next launch then starts
    // as these CTAs finish, and the block scheduler spreads its CTAs evenly over the
    // SMs (CTAs let in early fill the SMs that happen to finish first, up to five on
    // one SM, and the most crowded SM then sets the length of that launch).
    auto finish = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
        if (waiter) pdl_wait();
    };
    if (bad || other_class) {                                     // uniform across the CTA
        if (bad && tid == 0 && h == 0) atomicOr(a.status, bad);
        finish();
        return;
    }
    const int C = len + T;
    const int CP = round16(C);
    // [K;Q] K^T in two column ranges (rows 0..63 also in lanes 64..127) when every row
    // of [K;Q] fits in 64 lanes; else one MMA over all columns
    constexpr bool kSplitKK = CMAX + 16 <= 64;
    const int ca = !kSplitKK ? CP : CP == 16 ? 16 : ((CP / 2 + 15) & ~15);   // columns of the first MMA
    const size_t unit = static_cast<size_t>(slot) * H + h;
    const int ytile = static_cast<int>(unit) * 128;

    // ---- the buffered rows (keys, values, gates) of this unit
    const __nv_bfloat16 *bk = reinterpret_cast<const __nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
    const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
    __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(a.buf_k) + (unit * cap + len) * 128;
    __nv_bfloat16 *wv = reinterpret_cast<__nv_bfloat16 *>(a.buf_v) + (unit * cap + len) * 128;
    constexpr int NB = 4;                                         // rows 0 .. 31 in registers (T = 16:
    uint4 bkr[NB], bvr[NB];                                       // every buffered row); the rest below
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int r = dj + 8 * i;
        bkr[i] = make_uint4(0u, 0u, 0u, 0u);
        bvr[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < len) {
            bkr[i] = __ldg(reinterpret_cast<const uint4 *>(bk + static_cast<size_t>(r) * 128) + dc);
            bvr[i] = __ldg(reinterpret_cast<const uint4 *>(bv + static_cast<size_t>(r) * 128) + dc);
        }
    }
    float gq[P::NPL], bq[P::NPL];
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < P::NPL; ++i) {
            const int t = lane + 32 * i;
            gq[i] = 0.f;
            bq[i] = 0.f;
            if (t < len) {
                gq[i] = a.buf_g[unit * cap + t];
                bq[i] = a.buf_beta[unit * cap + t];
            }
            // draft token t - len sits in lane t - len (every lane takes part)
            const int src = t >= len && t < C ? t - len : 0;
            const float g2 = __shfl_sync(0xffffffffu, dg, src), b2 = __shfl_sync(0xffffffffu, db, src);
            if (t >= len && t < C) {
                gq[i] = g2;
                bq[i] = b2;
            }
        }
    }
    // ---- rows into the swizzled bf16 tiles: [K;Q] = buffered keys, draft keys, draft
    //      queries, then zeros; V = buffered values, draft values, then zeros.  The
    //      draft keys and values also go to the buffer (slots len .. len + T - 1).
    auto kq_at = [&](int r, int c) { return reinterpret_cast<uint4 *>(sKQ + (c >> 3) * P::SUBK + sw128(r, c & 7)); };
    auto v_at = [&](int r, int c) { return reinterpret_cast<uint4 *>(sV + (c >> 3) * P::SUBV + sw128(r, c & 7)); };
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int r = dj + 8 * i;
        if (r < len) {
            *kq_at(r, dc) = bkr[i];
            *v_at(r, dc) = bvr[i];
        }
    }
    for (int r = 8 * NB + dj; r < len; r += 8) {                  // longer buffers (drafts below 16)
        *kq_at(r, dc) = __ldg(reinterpret_cast<const uint4 *>(bk + static_cast<size_t>(r) * 128) + dc);
        *v_at(r, dc) = __ldg(reinterpret_cast<const uint4 *>(bv + static_cast<size_t>(r) * 128) + dc);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int j = dj + 8 * i;
        if (j < T) {
            *kq_at(len + j, dc) = draft[i];
            *kq_at(C + j, dc) = draft[2 + i];
            *v_at(len + j, dc) = draft[4 + i];
            reinterpret_cast<uint4 *>(wk + static_cast<size_t>(j) * 128)[dc] = draft[i];
            reinterpret_cast<uint4 *>(wv + static_cast<size_t>(j) * 128)[dc] = draft[4 + i];
        }
    }
#pragma unroll
    for (int i = 0; i < P::NPA / 8; ++i) {
        const int r = dj + 8 * i;
        if (r >= C + T) *kq_at(r, dc) = make_uint4(0u, 0u, 0u, 0u);
        if (r >= C && r < CMAX) *v_at(r, dc) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (warp == 0) {                                              // compensated scan of g
        float hi[P::NPL], lo[P::NPL];
#pragma unroll
        for (int i = 0; i < P::NPL; ++i) {
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
#pragma unroll
        for (int i = 1; i < P::NPL; ++i) {                        // carry the earlier columns' total
            const float chh = __shfl_sync(0xffffffffu, hi[i - 1], 31), cll = __shfl_sync(0xffffffffu, lo[i - 1], 31);
            const float s1 = hi[i] + chh, bp = s1 - hi[i];
            lo[i] += cll + ((hi[i] - (s1 - bp)) + (chh - bp));
            hi[i] = s1;
        }
#pragma unroll
        for (int i = 0; i < P::NPL; ++i) {
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
    if (tid == 0 && !expire) {                                    // [K;Q] K^T: coefficients
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) prefetch_tile_l2(&tm_state, q * 32, ytile);
        const uint64_t dkq = desc_sw128(kq0), dkq_up = desc_sw128(kq0 - 8192);
        const uint32_t idA = idesc_mn(1, 128, ca), idB = idesc_mn(1, 128, CP - ca);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {                          // lanes 0..127 = rows, columns [0, ca)
            const uint64_t d = desc_add(dkq, (ks >> 2) * P::SUBK + (ks & 3) * 32);
            mma_bf16(tmem, d, d, idA, ks > 0);
        }
        if (kSplitKK && CP > ca) {                                // lanes 64..127 = rows, columns [ca, CP)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * P::SUBK + (ks & 3) * 32;
                mma_bf16(tmem + ca, desc_add(dkq_up, off), desc_add(dkq, off + ca * 128), idB, ks > 0);
            }
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
    bool ok = !expire && mbar_wait(&bar[2], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            if (!expire && !mbar_wait(&bar[2], 0)) atomicOr(a.status, GDN_STATUS_DRAIN);
            atomicOr(a.status, kStatusTimeout);
        }
        finish();
        return;
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // ---- coefficient rows: row r of [K;Q] (TMEM lane r for columns [0, ca), lane
    //      64 + r for [ca, CP)); key rows t < C give A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s)
    //      (s < t), query rows C + t2 give M[t2][s] = e^{G_p-G_s} (q_t2.k_s) (s <= p);
    //      rows t2 >= T of M are zero; warps 0-1 write columns [0, ca), warps 2-3 the rest
    const int row = kSplitKK ? (tid & 63) : tid;
    if ((kSplitKK ? (warp & 1) : warp) * 32 < C + 16) {           // warp-uniform: the loads are collective
        const bool is_q = row >= C;
        const int t2 = row - C;
        const bool writes = row < C + 16;
        const bool live = row < C + T;
        const int p = !live ? C - 1 : is_q ? len + t2 : row;
        const float gh = sGh[p], gl = sGl[p];
        const float scl = is_q ? 1.f : sBeta[p];
        const int lim = !live ? 0 : is_q ? min(p + 1, C) : row;
        float *dst = is_q ? sMm + (writes ? t2 : 0) * CMAX : sAm + row * CMAX;
        const int cbeg = (!kSplitKK || warp < 2) ? 0 : ca, cend = (!kSplitKK || warp >= 2) ? CMAX : ca;
        const int r0 = (kSplitKK ? (warp & 1) : warp) * 32;         // the warp's first row
#pragma unroll 1
        for (int cb = 0; cb < CMAX / 16; ++cb) {                  // rolled: instruction fetch stalls lead
            const int c0 = cb * 16;
            if (c0 < cbeg || c0 >= cend) continue;                // warp-uniform
            // zeros for the whole warp (no exponentials; the stage is issue-bound): no
            // column below C, or only key rows, none of them past the block's first column
            const bool zero = c0 >= C || (r0 + 32 <= C && c0 >= r0 + 31);
            float mrow[16];
            if (zero) {
#pragma unroll
                for (int j = 0; j < 16; ++j) mrow[j] = 0.f;
            } else {
                float kq[16];
                tmem_ld16(lane_base + c0, kq);                    // c0 < C <= CP
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
            }
            if (writes) {
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4)
                    *reinterpret_cast<float4 *>(dst + c0 + 4 * j4) =
                        make_float4(mrow[4 * j4], mrow[4 * j4 + 1], mrow[4 * j4 + 2], mrow[4 * j4 + 3]);
            }
        }
    }
    tc_fence_before();                                            // K.K columns are reused by ve and O
    __syncthreads();
    // ---- W = M (I + A)^{-1}: warp w holds draft rows 4w .. 4w + 3, lane l token columns
    //      l, l + 32 (and l + 64); column s is final once every s' > s has been subtracted
    float x[P::NPL][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float *mr = sMm + (4 * warp + i) * CMAX;
#pragma unroll
        for (int j = 0; j < P::NPL; ++j) x[j][i] = lane + 32 * j < CMAX ? mr[lane + 32 * j] : 0.f;
    }
    // step s changes only the columns below s (A is strictly lower), so a step in token
    // group seg (columns 32 seg .. 32 seg + 31) updates the column groups 0 .. seg; the
    // stage is issue-bound with four CTAs on an SM, and the skipped updates were FMAs with
    // a zero A entry
#pragma unroll
    for (int seg = P::NPL - 1; seg >= 0; --seg) {
        const int s_top = (C < 32 * (seg + 1) ? C : 32 * (seg + 1)) - 1;
#pragma unroll 2
        for (int s = s_top; s >= 32 * seg; --s) {
            const float *ar = sAm + s * CMAX;
            float av[P::NPL];
#pragma unroll
            for (int j = 0; j <= seg; ++j) av[j] = lane + 32 * j < CMAX ? ar[lane + 32 * j] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = __shfl_sync(0xffffffffu, x[seg][i], s & 31);
#pragma unroll
                for (int j = 0; j <= seg; ++j) x[j][i] = fmaf(-w, av[j], x[j][i]);
            }
        }
    }
    __syncthreads();                                              // A, M no longer read: W goes over them
    // ---- W beta gamma and W beta as K-major [16][64] tiles, each the sum of two bf16
    //      terms (relative error 2^-16, far below that of the tf32 checkpoint product);
    //      token columns past 64 in [16][16] tiles with 32-byte swizzle
#pragma unroll
    for (int half = 0; half < P::NPL; ++half) {
        const int s = lane + 32 * half;
        if (s < CMAX) {
            const float bs = sBeta[s], bg = bs * sGam[s];
            const bool tail = P::TAIL && s >= 64;
            const uint32_t stride = tail ? 512 : 2048;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t2 = 4 * warp + i;
                const float w = x[half][i];
                __nv_bfloat16 t4[4];
                split2(w * bg, t4[0], t4[1]);
                split2(w * bs, t4[2], t4[3]);
                const uint32_t off = (tail ? 8192 + sw32(t2, (s - 64) >> 3) : sw128(t2, s >> 3)) + (s & 7) * 2;
#pragma unroll
                for (int j = 0; j < 4; ++j) *reinterpret_cast<__nv_bfloat16 *>(sW + j * stride + off) = t4[j];
            }
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {                                               // qe^T and ve^T, M = 128, N = 16
        tc_fence_after();
        const uint32_t idQ = idesc_mn(1, 128, 16) | kIdescMnMajorA;
        const int nks = CP / 16;
        const uint64_t dk = desc_mn_sw128(kq0, P::SUBK), dv = desc_mn_sw128(v0, P::SUBV), dw = desc_sw128(w0),
                       dwt = desc_sw32(w0 + 8192);
#pragma unroll
        for (int ks = 0; ks < CMAX / 16; ++ks) {
            if (ks < nks) {
                const uint64_t ak = desc_add(dk, ks * 2048), av = desc_add(dv, ks * 2048);
#pragma unroll
                for (int sp = 0; sp < 2; ++sp) {
                    const uint64_t wq = ks < 4 ? desc_add(dw, sp * 2048 + ks * 32) : desc_add(dwt, sp * 512);
                    const uint64_t wv = ks < 4 ? desc_add(dw, (2 + sp) * 2048 + ks * 32) : desc_add(dwt, (2 + sp) * 512);
                    mma_bf16(tmem + COL_Q, ak, wq, idQ, (sp | ks) != 0);
                    mma_bf16(tmem + COL_V, av, wv, idQ, (sp | ks) != 0);
                }
            }
        }
        mma_commit(&bar[3]);
    }
    ok = mbar_wait(&bar[3], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            if (!mbar_wait(&bar[3], 0)) atomicOr(a.status, GDN_STATUS_DRAIN);
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
        const uint64_t ds0 = desc_sw128(s00), dqe = desc_sw128(qe0);
        int loads[2] = {1, 1};                                    // TMA loads issued per buffer
        int mmas = 0;                                             // quarters whose MMAs were issued
        bool good = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int buf = q & 1;
            if (good && !mbar_wait(&bar[buf], q >> 1)) good = false;
            if (good) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_tf32(tmem + COL_O, desc_add(ds0, buf * 16384 + ks * 32), desc_add(dqe, q * 2048 + ks * 32),
                             idO, (q | ks) != 0);
                mma_commit(&bar[4 + q]);
                mmas = q + 1;
            }
            if (good && q < 2) {                                  // the buffer is reused once its MMAs are done
                if (!mbar_wait(&bar[4 + q], 0)) {
                    good = false;
                } else {
                    mbar_expect_tx(&bar[buf], 16384);
                    tma_load_2d(smem_raw + buf * 16384, &tm_state, (q + 2) * 32, ytile, &bar[buf]);
                    ++loads[buf];
                }
            }
        }
        if (!good) {                                              // wait (bounded) for what is in flight
            bool drained = true;
            for (int q = 0; q < mmas; ++q) drained &= mbar_wait(&bar[4 + q], 0);
            for (int i = 0; i < 2; ++i) drained &= mbar_wait(&bar[i], (loads[i] - 1) & 1);
            if (!drained) atomicOr(a.status, GDN_STATUS_DRAIN);
            *flag = 1;
        }
    }
    __syncthreads();
    ok = *flag == 0;
    if (ok) ok = mbar_wait(&bar[7], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            if (*flag == 0 && !mbar_wait(&bar[7], 0)) atomicOr(a.status, GDN_STATUS_DRAIN);
            atomicOr(a.status, kStatusTimeout);
        }
        finish();
        return;
    }
    pdl_release();                                                // the outputs are all that is left
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

// ---------------------------------------------------------------------------
// Fold (flush) through the inverse of the token system.
//
// For the L buffered tokens of one (sequence, head), with D_s = e^{G_{L-1}-G_s} and
// Tinv = (I + A)^{-1}, the checkpoint after the buffer is
//   S_L = gamma_{L-1} S0 + sum_s D_s u_s k_s^T,  u = Tinv r,  r_s = beta_s (v_s - gamma_s S0 k_s),
// and exchanging the sums gives S_L = gamma_{L-1} S0 + sum_s' (v_s' - gamma_s' S0 k_s') E'[s']
// with E'[s'] = beta_s' sum_s Tinv[s][s'] D_s k_s (L x d_k).  E' depends on the tokens
// only, so the triangular work happens on an L x L matrix, not per state row:
//   1. [K] K^T on the tensor cores (bf16 rows as loaded), A in shared memory;
//   2. Tinv by blocks of 16: the diagonal blocks by forward substitution (a thread
//      per column), the blocks below by T_ij = -T_ii sum_k A_ik T_kj, one block
//      diagonal at a time;
//   3. E'^T = K^T F^T with F[s'][s] = beta_s' D_s Tinv[s][s'] split into two bf16 terms,
//      the keys read as an MN-major operand;
//   4. S0 K^T in tf32, its checkpoint quarters streamed from L2 through two 16 KB
//      buffers while steps 1-2 run; R'[i][s] = -gamma_s (S0 k_s)[i] as two bf16 terms;
//   5. one M = 128, N = 128 contraction D = V^T E' + R' E' (values MN-major and exact;
//      hi.hi + hi.lo + lo.hi of the split terms, relative error about 2^-16, far below
//      that of the tf32 S0 K^T); S_L = gamma_{L-1} S0 + D row by row.
// Persistent: the CTAs list the sequences that flush (len >= threshold, or len > 0
// when forced) in the same order and take (sequence, head) items with a grid stride.
// DRAFT: the fused step; after the fold the CTA verifies the draft from S_L (the
// buffer is then empty) and stages it at buffer slot 0.
//
// Shared-memory plan (bytes from the 1024-aligned base), Lp = CMAX:
//   [OFF_AT, +Lp^2 4)      A^T, fp32 (row s holds column s of A)
//   [OFF_TI, +Lp^2 4)      Tinv, fp32 row-major; then the block scratch
//   [OFF_K, +2 SUBK)       key rows, bf16, 2 sub-tiles of CMAX rows x 128 B
//   [0, 32K)               after E' is formed: E'^T as two bf16 tiles [128][64]
//   [OFF_V, +2 SUBV)       value rows, bf16
//   [OFF_KF, +4 KFSUB)     key rows, fp32, 4 sub-tiles of CMAX rows x 128 B (S0 K^T);
//                          then F as two bf16 tiles [CMAX][64]
//   [OFF_Q, +32K)          the two checkpoint buffers; then R' as two bf16 tiles [128][64]
//   after the fold contraction: D, then S_L (rows, swizzled) in four 16 KB sub-tiles at
//   [0, 32K) and [OFF_Q, +32K); draft (DRAFT): its token tiles in the fp32 key region
//   (free once E' is formed) and qe over the value rows (free after the fold)
//   [OFF_SC, ...)          mbarriers, TMEM slot, flags, G (hi, lo), beta, gamma, D, list
// CMAX = 80: K K^T is one M = 128 MMA (rows 0..79 in lanes 0..79), and every operand
// whose K extent is the tokens holds tokens 64..79 in a second, 32-byte swizzled atom:
// F's at [OFF_KF + OFF_FT, +2 x 80 x 32), R''s at [OFF_KF + OFF_RT, +8K) (both free
// of the draft tiles), E'^T's at [OFF_ET, +8K) (over Tinv, read once F is formed).
template <int CMAX> struct FoldPlan {
    static constexpr bool SPLIT = CMAX <= 64;                 // K K^T rows in 64 lanes, twice
    static constexpr bool TAIL = CMAX > 64;
    static constexpr int NPL = (CMAX + 31) / 32;              // tokens per lane of warp 0
    static constexpr int SUBK = CMAX * 128;
    static constexpr int OFF_AT = 0;
    static constexpr int OFF_TI = OFF_AT + CMAX * CMAX * 4;
    static constexpr int OFF_Y = OFF_TI + CMAX * CMAX * 4;    // Tinv block scratch
    static constexpr int Y_END = OFF_Y + (CMAX / 16 - 1) * 1024;
    static constexpr int OFF_K = (Y_END + 1023) & ~1023;      // >= 8 KB: an operand may start 64 rows before
    static constexpr int K_END = OFF_K + 2 * SUBK;
    static constexpr int OFF_V = ((K_END > 32768 ? K_END : 32768) + 1023) & ~1023;
    static constexpr int SUBV = CMAX * 128;
    static constexpr int OFF_KF = OFF_V + 2 * SUBV;
    static constexpr int KFSUB = CMAX * 128;
    static constexpr int OFF_Q = OFF_KF + 4 * KFSUB;
    static constexpr int OFF_SC = OFF_Q + 32768;
    static constexpr int BYTES = OFF_SC + 160 + 20 * CMAX + 256;
    static constexpr int OFF_FT = 2 * CMAX * 128;             // from OFF_KF: F, tokens 64..79
    static constexpr int OFF_RT = (OFF_FT + 2 * CMAX * 32 + 1023) & ~1023;   // from OFF_KF: R', tokens 64..79
    static constexpr int OFF_ET = 32768;                      // E'^T, tokens 64..79
    static_assert(CMAX == 48 || CMAX == 64 || CMAX == 80, "token blocks");
    static_assert(!TAIL || (OFF_RT >= 22528 && OFF_RT + 8192 <= 4 * KFSUB), "R' tail past the draft tiles");
    static_assert(!TAIL || (OFF_ET >= OFF_TI && OFF_ET + 8192 <= OFF_V), "E' tail over Tinv, below the values");
    static_assert(OFF_K + SUBK + 16384 <= OFF_SC, "M = 128 operand reads stay inside the allocation");
    static_assert(OFF_K >= 8192 && K_END <= OFF_V, "64 rows of room before the keys; keys below the values");
    static_assert(2 * CMAX * 128 <= 4 * KFSUB, "F over the fp32 key tile");
    static_assert(4 * KFSUB >= 22528, "draft tiles in the fp32 key region");
    static_assert(2 * SUBV >= 8192, "draft qe tile over the value rows");
    static_assert(OFF_V >= 32768 && OFF_V + 2 * SUBV + 4 * KFSUB <= OFF_Q, "E^T tiles below the values");
    static_assert(OFF_SC >= 65536, "staging of the new state");
    static_assert((OFF_V % 1024) == 0 && (OFF_KF % 1024) == 0 && (OFF_Q % 1024) == 0 && (SUBK % 1024) == 0 &&
                  (KFSUB % 1024) == 0, "swizzle atoms");
};

template <int CMAX, bool DRAFT>
__global__ void __maxnreg__(kFoldRegs)
fold_eq_kernel(const __grid_constant__ CUtensorMap tm_state, const ReplayArgs a)
{
    using P = FoldPlan<CMAX>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, cap = a.cap;

    const bool expire = (a.flags & GDN_FLAG_TEST_EXPIRE) != 0;   // see the verify kernel

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (saddr(smem_raw) & 1023u) {
        if (tid == 0) atomicOr(a.status, kStatusTimeout);
        return;
    }
    uint8_t *sK = smem_raw + P::OFF_K;
    float *sAt = reinterpret_cast<float *>(smem_raw + P::OFF_AT);
    float *sTi = reinterpret_cast<float *>(smem_raw + P::OFF_TI);
    uint8_t *sEt = smem_raw;                                      // 2 x 16 KB
    uint8_t *sV = smem_raw + P::OFF_V;
    uint8_t *sKf = smem_raw + P::OFF_KF;
    uint8_t *sF = smem_raw + P::OFF_KF;                           // 2 x CMAX x 128 B, over the fp32 keys
    float *sY = reinterpret_cast<float *>(smem_raw + P::OFF_Y);   // [3][16][16]
    uint8_t *sBuf = smem_raw + P::OFF_Q;                          // 2 x 16 KB
    uint8_t *sR = smem_raw + P::OFF_Q;                            // 2 x 16 KB
    // the new state (D, then S_L), 4 sub-tiles of 16 KB: two over E'^T, two over R'
    auto snew = [&](int k) -> uint8_t * { return smem_raw + (k < 2 ? k * 16384 : P::OFF_Q + (k - 2) * 16384); };
    uint8_t *sm = smem_raw + P::OFF_SC;
    // 0: K.K; 1: E^T; 2, 3: checkpoint buffers; 4..7: S0 K^T quarters; 8: fold;
    // 9..11: draft (K_d K_d^T, qe/ve, S_L qe^T)
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 128);
    int *flag = reinterpret_cast<int *>(sm + 132);
    uint32_t *fmask = reinterpret_cast<uint32_t *>(sm + 144);     // [4]: folding sequences of a chunk
    float *sGh = reinterpret_cast<float *>(sm + 160);
    float *sGl = sGh + CMAX;
    float *sBeta = sGl + CMAX;
    float *sGam = sBeta + CMAX;
    float *sD = sGam + CMAX;
    float *dGh = sD + CMAX;      // draft: G (hi, lo), beta, gamma
    float *dGl = dGh + 16;
    float *dBeta = dGl + 16;
    float *dGam = dBeta + 16;
    // E' is read out before the fold contraction is issued into COL_F
    constexpr uint32_t COL_KK = 0, COL_E = P::TAIL ? 128 : 64, COL_P = 0, COL_F = 128;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 12; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_release();
    // TMEM is taken at the first item only: a CTA without one leaves the columns to
    // the kernels running beside this launch
    uint32_t tmem = 0, lane_base = 0;
    bool have_tmem = false;
    const uint32_t k0 = saddr(sK), f0 = saddr(sF), kf0 = saddr(sKf), buf0 = saddr(sBuf), r0 = saddr(sR),
                   e0 = saddr(sEt), v0 = saddr(sV);
    // base descriptors (issue sequences add constant offsets)
    const uint64_t dK = desc_sw128(k0), dKmn = desc_mn_sw128(k0, P::SUBK), dF = desc_sw128(f0),
                   dKf = desc_sw128(kf0), dBuf = desc_sw128(buf0), dR = desc_sw128(r0), dE = desc_sw128(e0),
                   dVmn = desc_mn_sw128(v0, P::SUBV);

    uint32_t it = 0;                                              // items done by this CTA
    bool alive = true;
    for (int b0 = 0; b0 < a.B && alive; b0 += kThreads) {
        // the folding sequences of this chunk of 128, identical in every CTA: one
        // ballot per warp; item n of the chunk is the n-th set bit over the four masks
        const int bb = b0 + tid;
        bool f = false;
        if (bb < a.B) {
            const int sl = a.state_idx ? a.state_idx[bb] : bb;
            if (sl >= 0 && sl < a.n_slot) {                         // others: reported by the length kernel
                const int ln = a.buf_len[sl];
                f = ln >= 0 && ln <= cap && (ln >= a.threshold || (a.force && ln > 0));
            }
        }
        const uint32_t m = __ballot_sync(0xffffffffu, f);
        __syncthreads();                                          // the previous chunk's masks are read
        if (lane == 0) fmask[warp] = m;
        __syncthreads();
        const uint32_t m0 = fmask[0], m1 = fmask[1], m2 = fmask[2], m3 = fmask[3];
        const int c1 = __popc(m0), c2 = c1 + __popc(m1), c3 = c2 + __popc(m2);
        const int n_items = (c3 + __popc(m3)) * H;
        for (int w = blockIdx.x; w < n_items && alive; w += gridDim.x, ++it) {
            if (!have_tmem) {                                     // uniform across the CTA
                if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                tmem = *tmem_slot;
                lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
                have_tmem = true;
            }
            const uint32_t ph = it & 1u;
            const int n = w / H, h = w % H;
            const int wi = n < c1 ? 0 : n < c2 ? 1 : n < c3 ? 2 : 3;
            const int b = b0 + wi * 32 +
                          static_cast<int>(__fns(wi == 0 ? m0 : wi == 1 ? m1 : wi == 2 ? m2 : m3, 0u,
                                                 n - (wi == 0 ? 0 : wi == 1 ? c1 : wi == 2 ? c2 : c3) + 1));
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
            static_assert(NV * kThreads == CMAX * 16, "token rows over the threads");
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
            // DRAFT: the draft rows are requested now, beside the buffered rows, and held in
            // registers until their tiles are free (after E' is formed)
            uint4 dkq[DRAFT ? 4 : 1], dvv[DRAFT ? 2 : 1];
            float dgq = 0.f, dbq = 0.f;
            if constexpr (DRAFT) {
                const int T = a.T;
                const size_t drow0 = (static_cast<size_t>(b) * T * H + h) * 128;
                const size_t dstride = static_cast<size_t>(H) * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15, t = r & 15;
                    dkq[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (t < T)
                        dkq[i] = __ldg(reinterpret_cast<const uint4 *>(
                                           reinterpret_cast<const __nv_bfloat16 *>(r < 16 ? a.k : a.q) + drow0 +
                                           static_cast<size_t>(t) * dstride) + c);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    dvv[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (r < T)
                        dvv[i] = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.v) +
                                                                       drow0 + static_cast<size_t>(r) * dstride) + c);
                }
                if (warp == 0 && lane < T) {
                    const size_t gi = (static_cast<size_t>(b) * T + lane) * H + h;
                    dgq = a.g[gi];
                    dbq = a.beta[gi];
                }
            }
            float gq[P::NPL], bq[P::NPL];
            if (warp == 0) {
#pragma unroll
                for (int i = 0; i < P::NPL; ++i) {
                    const int t = lane + 32 * i;
                    gq[i] = 0.f;
                    bq[i] = 0.f;
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
                float hi[P::NPL], lo[P::NPL];
#pragma unroll
                for (int i = 0; i < P::NPL; ++i) {
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
#pragma unroll
                for (int i = 1; i < P::NPL; ++i) {                // carry the earlier tokens' total
                    const float chh = __shfl_sync(0xffffffffu, hi[i - 1], 31);
                    const float cll = __shfl_sync(0xffffffffu, lo[i - 1], 31);
                    const float s1 = hi[i] + chh, bp = s1 - hi[i];
                    lo[i] += cll + ((hi[i] - (s1 - bp)) + (chh - bp));
                    hi[i] = s1;
                }
                // G_{L-1} (hi, lo) from the lane that holds it
                const int src = (L - 1) & 31, seg = (L - 1) >> 5;
                float sh = hi[0], sl = lo[0];
#pragma unroll
                for (int i = 1; i < P::NPL; ++i) {
                    sh = seg == i ? hi[i] : sh;
                    sl = seg == i ? lo[i] : sl;
                }
                const float gLh = __shfl_sync(0xffffffffu, sh, src);
                const float gLl = __shfl_sync(0xffffffffu, sl, src);
#pragma unroll
                for (int i = 0; i < P::NPL; ++i) {
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
            // thread 0 issues the token contractions; the S0 K^T pipeline (checkpoint quarters
            // from L2 through two buffers) is issued by thread 96, whose warp has no part in
            // the A^T and diagonal-block stages, so that it is complete by the time R' is formed
            constexpr int kPipe = 96;
            int loads[2] = {0, 0}, pk_mmas = 0;
            bool good = true;
            const uint32_t idP = idesc_mn(2, 128, Lp);
            auto pk_mma = [&](int q) {                            // thread kPipe: MMAs of quarter q
                const int bi = q & 1;
                if (good && !mbar_wait(&bar[2 + bi], q >> 1)) good = false;
                if (!good) return;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_tf32(tmem + COL_P, desc_add(dBuf, bi * 16384 + ks * 32), desc_add(dKf, q * P::KFSUB + ks * 32),
                             idP, (q | ks) != 0);
                mma_commit(&bar[4 + q]);
                pk_mmas = q + 1;
            };
            auto pk_load = [&](int q) {                           // thread kPipe: quarter q into buffer q & 1
                const int bi = q & 1;
                if (q >= 2 && good && !mbar_wait(&bar[4 + q - 2], ph)) good = false;
                if (!good) return;
                mbar_expect_tx(&bar[2 + bi], 16384);
                tma_load_2d(sBuf + bi * 16384, &tm_state, q * 32, ytile, &bar[2 + bi]);
                ++loads[bi];
            };
            // K K^T in two column ranges: lanes 0..63 hold rows 0..63 for columns [0, ca),
            // and, from an operand starting 64 rows before the key tile, lanes 64..127
            // hold rows 0..63 for columns [ca, Lp); all four warps then build A^T.
            // Beyond 64 tokens: one MMA, lane t = row t, three warps build A^T.
            const int ca = !P::SPLIT ? Lp : Lp == 16 ? 16 : ((Lp / 2 + 15) & ~15);
            if (tid == 0 && !expire) {                            // K K^T
                tc_fence_after();
                const uint32_t idA = idesc_mn(1, 128, ca), idB = idesc_mn(1, 128, Lp - ca);
                const uint64_t dKup = desc_sw128(k0 - 8192);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = desc_add(dK, (ks >> 2) * P::SUBK + (ks & 3) * 32);
                    mma_bf16(tmem + COL_KK, d, d, idA, ks > 0);
                }
                if (P::SPLIT && Lp > ca) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * P::SUBK + (ks & 3) * 32;
                        mma_bf16(tmem + COL_KK + ca, desc_add(dKup, off), desc_add(dK, off + ca * 128), idB, ks > 0);
                    }
                }
                mma_commit(&bar[0]);
            }
            if (tid == kPipe && !expire) {
                pk_load(0);
                pk_load(1);
            }
            bool ok = !expire && mbar_wait(&bar[0], ph);
            auto drain = [&]() {                                  // after a failed wait: what each issuer started
                bool drained = true;
                if (tid == 0 && !expire) drained &= mbar_wait(&bar[0], ph);
                if (tid == kPipe) {
                    for (int q = 0; q < pk_mmas; ++q) drained &= mbar_wait(&bar[4 + q], ph);
                    for (int i = 0; i < 2; ++i)
                        if (loads[i]) drained &= mbar_wait(&bar[2 + i], (loads[i] - 1) & 1);
                }
                if (!drained) atomicOr(a.status, GDN_STATUS_DRAIN);
                if (tid == 0) atomicOr(a.status, kStatusTimeout);
            };
            if (__syncthreads_or(!ok)) {
                drain();
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- A^T: thread t writes column t of A (row t of A^T): A[t][s] for s < t;
            //      warps 0-1 columns s in [0, ca), warps 2-3 the rest (token t = tid & 63);
            //      beyond 64 tokens, token t = tid over all columns
            if ((P::SPLIT ? (warp & 1) : warp) * 32 < CMAX) {     // warp-uniform: collective loads
                const int t = P::SPLIT ? (tid & 63) : tid;
                const float gh = t < L ? sGh[t] : 0.f, gl = t < L ? sGl[t] : 0.f, bt = t < L ? sBeta[t] : 0.f;
                const int cbeg = (!P::SPLIT || warp < 2) ? 0 : ca, cend = (!P::SPLIT || warp >= 2) ? CMAX : ca;
#pragma unroll 1
                for (int cb = 0; cb < CMAX / 16; ++cb) {
                    const int c0 = cb * 16;
                    if (c0 < cbeg || c0 >= cend) continue;        // warp-uniform
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
            tc_fence_before();
            __syncthreads();
            if (tid == kPipe) {                                   // during the diagonal blocks
                pk_mma(0);
                pk_mma(1);
                pk_load(2);
                pk_load(3);
            }
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
            if (tid == kPipe) {
                pk_mma(2);
                pk_mma(3);
                if (!good) *flag = 1;
            }
            __syncthreads();
            ok = *flag == 0;
            if (ok) ok = mbar_wait(&bar[7], ph);                  // S0 K^T complete: key and S0 tiles free
            if (__syncthreads_or(!ok)) {
                drain();
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- R'[d_v = tid][s] = -gamma_s (S0 k_s) as two bf16 terms (the value part of r
            //      enters the contraction directly: r_s = beta_s v_s + beta_s R'_s, and beta
            //      is folded into F)
#pragma unroll 1
            for (int cb = 0; cb < CMAX / 16; ++cb) {
                if (cb < nb) {
                    float pk[16];
                    tmem_ld16(lane_base + COL_P + cb * 16, pk);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const float4 g0 = *reinterpret_cast<const float4 *>(sGam + cb * 16 + 8 * hf);
                        const float4 g1 = *reinterpret_cast<const float4 *>(sGam + cb * 16 + 8 * hf + 4);
                        const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                        __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) split2(-gm[j] * pk[8 * hf + j], hh[j], ll[j]);
                        const bool tail = P::TAIL && cb >= 4;         // tokens 64..79
                        uint8_t *dst = tail ? sKf + P::OFF_RT + sw32(tid, hf) : sR + sw128(tid, 2 * cb + hf);
                        const uint32_t lo_off = tail ? 4096 : 16384;
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(
                            pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                        *reinterpret_cast<uint4 *>(dst + lo_off) = make_uint4(
                            pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
                    }
                }
            }
            // ---- F[s'][s] = beta_s' D_s Tinv[s][s'] as two bf16 K-major tiles [Lp][64] (over
            //      the fp32 key tile, no longer read); columns 64..79 in [Lp][16] tiles
            constexpr int NCH = P::TAIL ? 10 : 8;                 // 8-column chunks per row
            for (int e = tid; e < Lp * NCH; e += kThreads) {
                const int sp = e / NCH, c8 = e % NCH;             // row s', 8 columns s = 8 c8 ..
                const float bsp = sBeta[sp];
                __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int s = c8 * 8 + j;
                    const float v = s < CMAX ? bsp * sD[s] * sTi[s * CMAX + sp] : 0.f;
                    split2(v, hh[j], ll[j]);
                }
                const bool tail = P::TAIL && c8 >= 8;
                uint8_t *dst = tail ? sF + P::OFF_FT + sw32(sp, c8 - 8) : sF + sw128(sp, c8);
                const uint32_t lo_off = tail ? CMAX * 32 : CMAX * 128;
                *reinterpret_cast<uint4 *>(dst) =
                    make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]), pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                *reinterpret_cast<uint4 *>(dst + lo_off) =
                    make_uint4(pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {                                       // E^T = K^T F^T (keys MN-major)
                tc_fence_after();
                const uint32_t idE = idesc_mn(1, 128, Lp) | kIdescMnMajorA;
                const uint64_t dFt = desc_sw32(f0 + P::OFF_FT);
#pragma unroll
                for (int ks = 0; ks < CMAX / 16; ++ks) {
                    if (ks < nb) {
                        const uint64_t ak = desc_add(dKmn, ks * 2048);
                        const uint64_t fh = ks < 4 ? desc_add(dF, ks * 32) : dFt;
                        const uint64_t fl = ks < 4 ? desc_add(dF, CMAX * 128 + ks * 32) : desc_add(dFt, CMAX * 32);
                        mma_bf16(tmem + COL_E, ak, fh, idE, ks > 0);
                        mma_bf16(tmem + COL_E, ak, fl, idE, 1);
                    }
                }
                mma_commit(&bar[1]);
            }
            ok = mbar_wait(&bar[1], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    if (!mbar_wait(&bar[1], ph)) atomicOr(a.status, GDN_STATUS_DRAIN);
                    atomicOr(a.status, kStatusTimeout);
                }
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- E^T row d_k = tid as two bf16 terms, K-major [128][64] tiles
#pragma unroll 1
            for (int cb = 0; cb < CMAX / 16; ++cb) {
                if (cb < nb) {
                    float ev[16];
                    tmem_ld16(lane_base + COL_E + cb * 16, ev);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        __nv_bfloat16 hh[8], ll[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) split2(ev[8 * hf + j], hh[j], ll[j]);
                        const bool tail = P::TAIL && cb >= 4;         // tokens 64..79
                        uint8_t *dst = tail ? smem_raw + P::OFF_ET + sw32(tid, hf) : sEt + sw128(tid, 2 * cb + hf);
                        const uint32_t lo_off = tail ? 4096 : 16384;
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(pack2(hh[0], hh[1]), pack2(hh[2], hh[3]),
                                                                     pack2(hh[4], hh[5]), pack2(hh[6], hh[7]));
                        *reinterpret_cast<uint4 *>(dst + lo_off) = make_uint4(
                            pack2(ll[0], ll[1]), pack2(ll[2], ll[3]), pack2(ll[4], ll[5]), pack2(ll[6], ll[7]));
                    }
                }
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {                                       // D = V^T E' + R' E'
                tc_fence_after();
                const uint32_t idF = idesc_mn(1, 128, 128), idV = idF | kIdescMnMajorA;
                const uint64_t dRt = desc_sw32(kf0 + P::OFF_RT), dEt = desc_sw32(saddr(smem_raw) + P::OFF_ET);
#pragma unroll
                for (int ks = 0; ks < CMAX / 16; ++ks) {
                    if (ks < nb) {
                        const uint64_t av = desc_add(dVmn, ks * 2048);
                        const uint64_t rh = ks < 4 ? desc_add(dR, ks * 32) : dRt;
                        const uint64_t rl = ks < 4 ? desc_add(dR, 16384 + ks * 32) : desc_add(dRt, 4096);
                        const uint64_t eh = ks < 4 ? desc_add(dE, ks * 32) : dEt;
                        const uint64_t el = ks < 4 ? desc_add(dE, 16384 + ks * 32) : desc_add(dEt, 4096);
                        mma_bf16(tmem + COL_F, av, eh, idV, ks > 0);
                        mma_bf16(tmem + COL_F, av, el, idV, 1);
                        mma_bf16(tmem + COL_F, rh, eh, idF, 1);
                        mma_bf16(tmem + COL_F, rh, el, idF, 1);
                        mma_bf16(tmem + COL_F, rl, eh, idF, 1);
                    }
                }
                mma_commit(&bar[8]);
            }
            // ---- DRAFT (fused step): the draft is then verified from S_L (the buffer is
            //      empty after the fold) by effective queries over the 16 draft tokens alone
            //      (G' restarted at the draft): W' = M' (I + A')^{-1}, qe = gamma' q - (W' beta'
            //      gamma') K_d, ve = (W' beta') V_d, o = scale (S_L qe + ve).  Everything but the
            //      S_L contraction runs while the fold contraction executes; its tiles sit in
            //      the fp32 key region (free since E' was formed), its accumulators in the TMEM
            //      columns of S0 K^T.  The draft is staged at buffer slot 0.
            constexpr int SUBKD = 4096, SUBVD = 2048;             // [K_d; Q_d] 32 rows, V_d 16 rows
            uint8_t *sDKQ = sKf;                                  // 2 sub-tiles of 32 rows x 128 B
            uint8_t *sVd = sKf + 8192;                            // 2 sub-tiles of 16 rows x 128 B
            float *sAd = reinterpret_cast<float *>(sKf + 12288);  // A' [16][16]
            float *sMd = sAd + 256;                               // M' [16][16]
            uint8_t *sWd = sKf + 14336;                           // W' beta' gamma', W' beta': 2 + 2 tiles [16][64]
            uint8_t *sQd = sV;                                    // qe, fp32 [16][128], after the fold
            constexpr uint32_t COL_KD = 0, COL_DQ = 16, COL_DV = 32, COL_DO = 48;
            if constexpr (DRAFT) {
                const int T = a.T;
                __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(a.buf_k) + unit * cap * 128;
                __nv_bfloat16 *wv = reinterpret_cast<__nv_bfloat16 *>(a.buf_v) + unit * cap * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    *reinterpret_cast<uint4 *>(sDKQ + (c >> 3) * SUBKD + sw128(r, c & 7)) = dkq[i];
                    if (r < T) reinterpret_cast<uint4 *>(wk + static_cast<size_t>(r) * 128)[c] = dkq[i];
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int e = tid + i * kThreads, r = e >> 4, c = e & 15;
                    *reinterpret_cast<uint4 *>(sVd + (c >> 3) * SUBVD + sw128(r, c & 7)) = dvv[i];
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
                __syncthreads();
                if (tid == 0) {                                   // [K_d; Q_d] K_d^T
                    tc_fence_after();
                    const uint32_t idK = idesc_mn(1, 128, 16);
                    const uint64_t dkd = desc_sw128(saddr(sDKQ));
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t d = desc_add(dkd, (ks >> 2) * SUBKD + (ks & 3) * 32);
                        mma_bf16(tmem + COL_KD, d, d, idK, ks > 0);
                    }
                    mma_commit(&bar[9]);
                }
                ok = mbar_wait(&bar[9], ph);
                if (__syncthreads_or(!ok)) {
                    if (tid == 0) {
                        const bool d8 = mbar_wait(&bar[8], ph), d9 = mbar_wait(&bar[9], ph);
                        if (!(d8 && d9)) atomicOr(a.status, GDN_STATUS_DRAIN);
                        atomicOr(a.status, kStatusTimeout);
                    }
                    alive = false;
                    break;
                }
                tc_fence_after();
                if (warp == 0) {                                  // lanes 0..15: A' rows, 16..31: M' rows
                    float kq[16];
                    tmem_ld16(lane_base + COL_KD, kq);
                    const bool is_q = lane >= 16;
                    const int t = lane & 15;
                    const float gh = dGh[t], gl = dGl[t], scl = is_q ? 1.f : dBeta[t];
                    const int lim = t >= T ? 0 : is_q ? t + 1 : t;
                    float *dst = (is_q ? sMd : sAd) + t * 16;
                    float mrow[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float e = __expf((gh - dGh[j]) + (gl - dGl[j]));
                        mrow[j] = j < lim ? scl * e * kq[j] : 0.f;
                    }
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        *reinterpret_cast<float4 *>(dst + 4 * j4) =
                            make_float4(mrow[4 * j4], mrow[4 * j4 + 1], mrow[4 * j4 + 2], mrow[4 * j4 + 3]);
                }
                __syncthreads();
                {                                                 // W' rows 4 warp .. 4 warp + 3, lane = column
                    float xw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) xw[i] = lane < 16 ? sMd[(4 * warp + i) * 16 + lane] : 0.f;
                    for (int s2 = T - 1; s2 >= 0; --s2) {
                        const float av = lane < 16 ? sAd[s2 * 16 + lane] : 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float w = __shfl_sync(0xffffffffu, xw[i], s2);
                            xw[i] = fmaf(-w, av, xw[i]);
                        }
                    }
                    if (lane < 16) {
                        const float bs = dBeta[lane], bg = bs * dGam[lane];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            __nv_bfloat16 t4[4];
                            split2(xw[i] * bg, t4[0], t4[1]);
                            split2(xw[i] * bs, t4[2], t4[3]);
                            const uint32_t off = sw128(4 * warp + i, lane >> 3) + (lane & 7) * 2;
#pragma unroll
                            for (int j = 0; j < 4; ++j) *reinterpret_cast<__nv_bfloat16 *>(sWd + j * 2048 + off) = t4[j];
                        }
                    }
                }
                fence_proxy_async();
                __syncthreads();
                if (tid == 0) {                                   // qe^T, ve^T (K_d, V_d MN-major)
                    tc_fence_after();
                    const uint32_t idQ = idesc_mn(1, 128, 16) | kIdescMnMajorA;
                    const uint64_t ak = desc_mn_sw128(saddr(sDKQ), SUBKD), av = desc_mn_sw128(saddr(sVd), SUBVD);
                    const uint64_t dw = desc_sw128(saddr(sWd));
                    mma_bf16(tmem + COL_DQ, ak, dw, idQ, 0);
                    mma_bf16(tmem + COL_DQ, ak, desc_add(dw, 2048), idQ, 1);
                    mma_bf16(tmem + COL_DV, av, desc_add(dw, 4096), idQ, 0);
                    mma_bf16(tmem + COL_DV, av, desc_add(dw, 6144), idQ, 1);
                    mma_commit(&bar[10]);
                }
            }
            // rows 32 warp .. 32 warp + 31 of S0 (L2), 512 contiguous bytes per warp load,
            // while the contraction runs
            float4 *srow = reinterpret_cast<float4 *>(a.state_out + (unit * 128 + 32 * warp) * 128) + lane;
            float4 x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = srow[i * 32];
            ok = mbar_wait(&bar[8], ph);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    bool drained = mbar_wait(&bar[8], ph);
                    if (DRAFT) drained &= mbar_wait(&bar[10], ph);
                    if (!drained) atomicOr(a.status, GDN_STATUS_DRAIN);
                    atomicOr(a.status, kStatusTimeout);
                }
                alive = false;
                break;
            }
            tc_fence_after();
            // ---- D row tid into shared memory (swizzled rows), then S_L = gamma_{L-1} S0 + D
            //      row by row with coalesced loads and stores
            // The fused kernel keeps both loops below rolled (its instruction footprint is the
            // larger; measured fused step 28.5 -> 27.6 us/layer); the flush kernel unrolls them
            // (rolled, its half-row loop holds both halves of the rows live and spills).
            auto stage_d = [&](int c0) {
                float dd[16];
                tmem_ld16(lane_base + COL_F + c0, dd);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = c0 + 4 * q;
                    *reinterpret_cast<float4 *>(snew(col >> 5) + sw128(tid, (col & 31) >> 2)) =
                        make_float4(dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
                }
            };
            if constexpr (DRAFT) {
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 16) stage_d(c0);
            } else {
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 16) stage_d(c0);
            }
            __syncwarp();                                         // a warp reads back only its own rows
            {
                const float gL = sGam[L - 1];
                const uint8_t *dsub = snew(lane >> 3);
                float4 x2[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x2[i] = srow[(16 + i) * 32];
                auto new_rows = [&](int hf) {
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
                };
                if constexpr (DRAFT) {
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) new_rows(hf);
                } else {
                    new_rows(0);
                    new_rows(1);
                }
            }
            if constexpr (DRAFT) {
                const int T = a.T;
                ok = mbar_wait(&bar[10], ph);
                if (__syncthreads_or(!ok)) {
                    if (tid == 0) {
                        if (!mbar_wait(&bar[10], ph)) atomicOr(a.status, GDN_STATUS_DRAIN);
                        atomicOr(a.status, kStatusTimeout);
                    }
                    alive = false;
                    break;
                }
                tc_fence_after();
                {                                                 // qe[t2][d_k = tid], fp32 K-major tile
                    float dq[16];
                    tmem_ld16(lane_base + COL_DQ, dq);
                    uint8_t *col = sQd + (tid >> 5) * 2048 + (tid & 3) * 4;
                    const uint8_t *qsrc = sDKQ + (tid >> 6) * SUBKD + (tid & 7) * 2;
#pragma unroll
                    for (int t2 = 0; t2 < 16; ++t2) {
                        const float qv = __bfloat162float(
                            *reinterpret_cast<const __nv_bfloat16 *>(qsrc + sw128(16 + t2, (tid & 63) >> 3)));
                        const float v = t2 < T ? fmaf(dGam[t2], qv, -dq[t2]) : 0.f;
                        *reinterpret_cast<float *>(col + sw128(t2, (tid & 31) >> 2)) = v;
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncthreads();
                if (tid == 0) {                                   // O = S_L qe^T (S_L from the staging tile)
                    tc_fence_after();
                    const uint32_t idO = idesc_mn(2, 128, 16);
                    const uint64_t dsa = desc_sw128(saddr(snew(0))), dsb = desc_sw128(saddr(snew(2)));
                    const uint64_t dqd = desc_sw128(saddr(sQd));
#pragma unroll
                    for (int ks = 0; ks < 16; ++ks)
                        mma_tf32(tmem + COL_DO, desc_add(ks < 8 ? dsa : dsb, ((ks >> 2) & 1) * 16384 + (ks & 3) * 32),
                                 desc_add(dqd, (ks >> 2) * 2048 + (ks & 3) * 32), idO, ks > 0);
                    mma_commit(&bar[11]);
                }
                ok = mbar_wait(&bar[11], ph);
                if (__syncthreads_or(!ok)) {
                    if (tid == 0) {
                        if (!mbar_wait(&bar[11], ph)) atomicOr(a.status, GDN_STATUS_DRAIN);
                        atomicOr(a.status, kStatusTimeout);
                    }
                    alive = false;
                    break;
                }
                tc_fence_after();
                float o[16], ve[16];
                tmem_ld16(lane_base + COL_DO, o);
                tmem_ld16(lane_base + COL_DV, ve);
#pragma unroll
                for (int t2 = 0; t2 < 16; ++t2)
                    if (t2 < T)
                        a.out[((static_cast<size_t>(b) * T + t2) * H + h) * 128 + tid] = a.scale * (o[t2] + ve[t2]);
            }
            tc_fence_before();
            __syncthreads();                                      // the tiles are reused by the next item
        }
        __syncthreads();                                          // the list is rebuilt
    }
    tc_fence_before();
    __syncthreads();
    if (have_tmem && warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int CMAX>
int launch_eq(const gdn_replay_dims *d, const ReplayArgs &a, const CUtensorMap &m, cudaStream_t s) {
    constexpr int smem = EqPlan<CMAX>::BYTES;
    auto kern = verify_eq_kernel<CMAX>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    return launch_pdl(kern, dim3(d->H, d->B), dim3(kThreads), smem, s, m, a) == cudaSuccess ? GDN_OK
                                                                                       : GDN_ERR_LAUNCH;
}

// Persistent fold launch: as many CTAs as fit at once (two per SM below 113 KB of
// shared memory; the 224-register cap allows two), at most one per (sequence, head).
template <bool DRAFT>
int launch_fold(const gdn_replay_dims *d, const ReplayArgs &a, const CUtensorMap &m, cudaStream_t s) {
    const int smem = d->cap <= 48 ? FoldPlan<48>::BYTES : d->cap <= 64 ? FoldPlan<64>::BYTES : FoldPlan<80>::BYTES;
    auto kern = d->cap <= 48 ? fold_eq_kernel<48, DRAFT> : d->cap <= 64 ? fold_eq_kernel<64, DRAFT>
                                                                        : fold_eq_kernel<80, DRAFT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int sms = sm_count();
    if (sms <= 0) return GDN_ERR_LAUNCH;
    int ctas = sms * ((smem + 1024) * 2 <= 228 * 1024 ? 2 : 1);
    ctas = ctas < d->B * d->H ? ctas : d->B * d->H;
    return launch_pdl(kern, dim3(ctas), dim3(kThreads), smem, s, m, a) == cudaSuccess ? GDN_OK
                                                                                 : GDN_ERR_LAUNCH;
}

}  // namespace

bool tc_shape(const gdn_replay_dims *d) {
    return d->dk == 128 && d->dv == 128 && d->in_dtype == GDN_DTYPE_BF16 && d->T <= 16 && d->cap <= 80;
}

int tc_verify(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    if (!tc_shape(d)) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_in, d->n_slot * d->H * 128)) return GDN_ERR_LAUNCH;
    return d->cap <= 48 ? launch_eq<48>(d, a, m, s) : d->cap <= 64 ? launch_eq<64>(d, a, m, s)
                                                                   : launch_eq<80>(d, a, m, s);
}

int tc_flush(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    if (!tc_shape(d)) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_out, d->n_slot * d->H * 128)) return GDN_ERR_LAUNCH;
    return launch_fold<false>(d, a, m, s);
}

int tc_verify_fold(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    if (!tc_shape(d)) return 1;
    CUtensorMap m;
    if (!state_map(&m, a.state_out, d->n_slot * d->H * 128)) return GDN_ERR_LAUNCH;
    ReplayArgs af = a;                                            // fold the full buffers, verify the draft
    af.force = 0;
    const int rc = launch_fold<true>(d, af, m, s);
    if (rc) return rc;
    ReplayArgs an = a;                                            // the rest, beside the fold launch
    an.fold_class = 1;
    return d->cap <= 48 ? launch_eq<48>(d, an, m, s) : d->cap <= 64 ? launch_eq<64>(d, an, m, s)
                                                                    : launch_eq<80>(d, an, m, s);
}

}  // namespace gdn
