// gla_tc.cu -- tcgen05 / TMEM / TMA chunk-wise prefill kernel for sm_103a.
//
// Method ("Gated Linear Attention", GLA Recurrent Form and Chunk-Wise
// Block-Parallel): S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t,
// evaluated 64 tokens at a time.  Unrolling the recurrence over one chunk
// ("linear-attention" blog, Gated linear attention: a write at i reaches t
// weighted by the product of alpha over (i, t]) and writing b_t for the
// inclusive cumsum of log alpha from the chunk start, b_C for its last value:
//   Qh_t = q_t * e^{b_t - b_C}        (>= 1 factor)
//   Kh_i = k_i * e^{b_C - b_i}        (<= 1 factor)
//   S'   = Diag(e^{b_C}) S_prev                      (decay first)
//   o_t  = Qh_t^T S' + sum_{i<=t} (Qh_t . Kh_i) v_i    (inter + intra)
//   S    = S' + Kh^T V
// which is exactly the recurrence, since (Qh_t . Kh_i) carries e^{b_t - b_i}.
//
// One CTA owns one (batch*head, 128-column slice of d_v) for the whole
// sequence.  The state is kept TRANSPOSED in tensor memory, S^T (lane = value
// column j, column = key channel d, fp32), so that every state/output
// product has M = 128 value columns:
//   MMA_A   A[t][i]  = Qh Kh^T            M=128 (rows 64..127 unused), N=64, K=dk
//   MMA_dS  S^T     += V^T Kh             M=128, N=dk, K=64      (V, Kh MN-major)
//   MMA_Oi  O^T      = S'^T_bf16 Qh^T     M=128, N=64, K=dk      (A from TMEM)
//   MMA_Oa  O^T     += V^T P^T            M=128, N=64, K=64      (P = tril(A), bf16)
// Warp roles (16 warps): 0-3 gate (cumsum + factors, in place on the q/k
// tiles), 4-7 state (decay S^T, write the bf16 copy), 8-11 output (O^T ->
// global), 12-13 P (mask A -> bf16 P in shared memory), 14 TMA producer,
// 15 MMA issuer and TMEM owner.  Every pipeline wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int C = 64;      // chunk length (tokens)
constexpr int DVT = 128;   // value columns per CTA (MMA M)
constexpr int NS = 3;      // q/k stages (hold Qh/Kh until the chunk's MMAs finish)
constexpr int NL = 2;      // log-alpha stages
constexpr int NV = 2;      // v stages
constexpr int kThreads = 512;

constexpr int W_STATE0 = 4, W_OUT0 = 8, W_P0 = 12, W_TMA = 14, W_MMA = 15;

// tensor-memory column map (512 columns allocated)
constexpr uint32_t TM_S = 0;     // S^T fp32, dk columns
constexpr uint32_t TM_SB = 128;  // 2 x bf16 copies of S'^T, dk/2 columns each
constexpr uint32_t TM_O = 256;   // 2 x O^T fp32, 64 columns each
constexpr uint32_t TM_A = 384;   // 2 x A fp32, 64 columns each
constexpr uint32_t TM_COLS = 512;

enum {
    B_QK_FULL = 0,
    B_QK_GATED = B_QK_FULL + NS,
    B_QK_EMPTY = B_QK_GATED + NS,
    B_LA_FULL = B_QK_EMPTY + NS,
    B_LA_EMPTY = B_LA_FULL + NL,
    B_V_FULL = B_LA_EMPTY + NL,
    B_V_EMPTY = B_V_FULL + NV,
    B_A_FULL = B_V_EMPTY + NV,
    B_A_EMPTY = B_A_FULL + 2,
    B_P_FULL = B_A_EMPTY + 2,
    B_P_EMPTY = B_P_FULL + 2,
    B_S_READY = B_P_EMPTY + 2,
    B_S_FULL = B_S_READY + 1,
    B_O_FULL = B_S_FULL + 1,
    B_O_EMPTY = B_O_FULL + 2,
    B_DRAIN = B_O_EMPTY + 2,
    B_COUNT = B_DRAIN + 1
};

template <int DK>
struct Layout {
    static constexpr int QB = DK * C * 2;          // one bf16 [64][DK] tile (DK/64 swizzle atoms)
    static constexpr int STAGE_QK = 2 * QB;
    static constexpr int LAB = DK * C * 4;         // fp32 [64][DK]
    static constexpr int VB = DVT * C * 2;         // bf16 [64][128] as two 64-column atoms
    static constexpr int PB = C * C * 2;           // bf16 [64][64]
    static constexpr int SEG = 128 / (DK / 2);     // token segments in the gate mapping
    static constexpr int off_qk = 0;
    static constexpr int off_la = off_qk + NS * STAGE_QK;
    static constexpr int off_v = off_la + NL * LAB;
    static constexpr int off_p = off_v + NV * VB;
    static constexpr int off_gamma = off_p + 2 * PB;
    static constexpr int off_segtot = off_gamma + NS * DK * 4;
    static constexpr int off_den = off_segtot + 2 * SEG * DK * 4;
    static constexpr int off_bar = off_den + 2 * C * 4;
    static constexpr int off_misc = off_bar + B_COUNT * 8;
    static constexpr int total = off_misc + 16;
    static constexpr int alloc = total + 1024;
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_la, tm_v;
    const float* init_state;
    const float* init_z;
    void* out;
    float* final_state;
    float* final_z;
    unsigned* err;
    int L, dv, nchunks, ntile;
    unsigned flags;
    int out_f32;
};

template <int DK, bool GATE>
__global__ void __launch_bounds__(kThreads, 1) gla_prefill_tc_kernel(const __grid_constant__ TcParams p) {
    using Ly = Layout<DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::off_bar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Ly::off_misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Ly::off_misc + 4);
    float* gamma = reinterpret_cast<float*>(sm + Ly::off_gamma);
    float* segtot = reinterpret_cast<float*>(sm + Ly::off_segtot);
    float* den = reinterpret_cast<float*>(sm + Ly::off_den);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x % p.ntile;
    const int bh = blockIdx.x / p.ntile;
    const int j0 = tile * DVT;
    const int L = p.L, dv = p.dv, N = p.nchunks;
    const bool norm = p.flags & GLA_FLAG_NORMALIZE;
    const bool elu = p.flags & GLA_FLAG_FEATURE_ELU1;
    // value lanes holding real columns; with the normaliser (dv == 64) lane 64 holds z
    const int jvalid = min(DVT, dv - j0);
    const int nvb = jvalid / 64;  // TMA-loaded 64-column blocks of V

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(bar(B_QK_FULL + i), 1);
            mbar_init(bar(B_QK_GATED + i), 4);
            mbar_init(bar(B_QK_EMPTY + i), 1);
        }
        for (int i = 0; i < NL; i++) {
            mbar_init(bar(B_LA_FULL + i), 1);
            mbar_init(bar(B_LA_EMPTY + i), 4);
        }
        for (int i = 0; i < NV; i++) {
            mbar_init(bar(B_V_FULL + i), 1);
            mbar_init(bar(B_V_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_A_FULL + i), 1);
            mbar_init(bar(B_A_EMPTY + i), 2);
            mbar_init(bar(B_P_FULL + i), 2);
            mbar_init(bar(B_P_EMPTY + i), 1);
            mbar_init(bar(B_O_FULL + i), 1);
            mbar_init(bar(B_O_EMPTY + i), 4);
        }
        mbar_init(bar(B_S_READY), 4);
        mbar_init(bar(B_S_FULL), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    // V columns the TMA never writes: zero, plus the all-ones normaliser column
    if (nvb < 2) {
        for (int idx = threadIdx.x; idx < NV * C * 64; idx += kThreads) {
            const int st = idx / (C * 64), rem = idx % (C * 64);
            const int row = rem / 64, col = rem % 64;
            const float x = (norm && col == 0) ? 1.f : 0.f;
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(sm + Ly::off_v + st * Ly::VB + 8192 +
                                                                  sw128_offset(row, col));
            *dst = __float2bfloat16_rn(x);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_field = static_cast<uint32_t>((warp & 3) * 32) << 16;

    // track outstanding TMA loads for the teardown (producer lane only)
    int last_issued = -1;

    if (warp < 4) {
        // ============================================================ gate
        constexpr int PAIRS = DK / 2;
        constexpr int SEG = Ly::SEG;
        constexpr int TPS = C / SEG;
        const int gt = threadIdx.x;
        const int pr = gt % PAIRS, h = gt / PAIRS;
        const int ch = 2 * pr;
        const int atom = ch >> 6, col = ch & 63;
        for (int c = 0; c < N; c++) {
            const int s = c % NS, l = c % NL;
            bool ok = true;
            if (GATE) ok = mbar_wait(bar(B_LA_FULL + l), (c / NL) & 1, abort_flag, p.err);
            if (ok) ok = mbar_wait(bar(B_QK_FULL + s), (c / NS) & 1, abort_flag, p.err);
            if (!GATE && !__all_sync(0xffffffffu, ok)) break;
            uint8_t* qt = sm + Ly::off_qk + s * Ly::STAGE_QK + atom * 8192;
            uint8_t* kt = qt + Ly::QB;
            const int nval = min(C, L - c * C);
            float b0[TPS], b1[TPS];
            float off0 = 0.f, off1 = 0.f, tot0 = 0.f, tot1 = 0.f;
            if (GATE) {
                const float* la = reinterpret_cast<const float*>(sm + Ly::off_la + l * Ly::LAB);
                float r0 = 0.f, r1 = 0.f;
                float* st = segtot + (c & 1) * SEG * DK;
                if (ok) {
#pragma unroll
                    for (int i = 0; i < TPS; i++) {
                        const float2 x = *reinterpret_cast<const float2*>(la + (h * TPS + i) * DK + ch);
                        r0 += x.x;
                        r1 += x.y;
                        b0[i] = r0;
                        b1[i] = r1;
                    }
                    st[h * DK + ch] = r0;
                    st[h * DK + ch + 1] = r1;
                }
                // exchange of segment totals doubles as the gate role's agreement to go on
                if (!bar_red_and(1, 128, ok)) break;
#pragma unroll
                for (int g = 0; g < SEG; g++) {
                    const float u0 = st[g * DK + ch], u1 = st[g * DK + ch + 1];
                    if (g < h) {
                        off0 += u0;
                        off1 += u1;
                    }
                    tot0 += u0;
                    tot1 += u1;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_LA_EMPTY + l));
                if (h == 0) {
                    gamma[s * DK + ch] = __expf(tot0);
                    gamma[s * DK + ch + 1] = __expf(tot1);
                }
            }
            if (GATE || elu || nval < C) {
#pragma unroll
                for (int i = 0; i < TPS; i++) {
                    const int t = h * TPS + i;
                    const uint32_t o = sw128_offset(t, col);
                    uint32_t* qp = reinterpret_cast<uint32_t*>(qt + o);
                    uint32_t* kp = reinterpret_cast<uint32_t*>(kt + o);
                    float2 qv = unpack_bf16x2(*qp), kv = unpack_bf16x2(*kp);
                    if (elu) {
                        qv.x = elu1(qv.x);
                        qv.y = elu1(qv.y);
                        kv.x = elu1(kv.x);
                        kv.y = elu1(kv.y);
                    }
                    if (GATE) {
                        const float d0 = (b0[i] + off0) - tot0;  // b_t - b_C >= 0
                        const float d1 = (b1[i] + off1) - tot1;
                        qv.x *= __expf(d0);
                        qv.y *= __expf(d1);
                        kv.x *= __expf(-d0);
                        kv.y *= __expf(-d1);
                    }
                    if (t >= nval) {  // padding tokens must not write the state (elu(0)+1 != 0)
                        qv = make_float2(0.f, 0.f);
                        kv = make_float2(0.f, 0.f);
                    }
                    *qp = pack_bf16x2(qv.x, qv.y);
                    *kp = pack_bf16x2(kv.x, kv.y);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QK_GATED + s));
        }
    } else if (warp < W_OUT0) {
        // ============================================================ state
        const int j = threadIdx.x - W_STATE0 * 32;
        const uint32_t tS = tmem + lane_field + TM_S;
        const float* s0 = p.init_state ? p.init_state + (long)bh * DK * dv + j0 + j : nullptr;
        for (int g = 0; g < DK / 32; g++) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; i++) {
                float x = 0.f;
                const int d = g * 32 + i;
                if (j < jvalid) {
                    if (s0) x = s0[(long)d * dv];
                } else if (norm && j == 64 && p.init_z) {
                    x = p.init_z[(long)bh * DK + d];
                }
                r[i] = __float_as_uint(x);
            }
            tmem_st32(tS + g * 32, r);
        }
        tmem_wait_st();
        bool ok = true;
        for (int c = 0; c < N && ok; c++) {
            const int s = c % NS;
            if (GATE && !mbar_wait_warp(bar(B_QK_GATED + s), (c / NS) & 1, abort_flag, p.err)) { ok = false; break; }
            if (c > 0 && !mbar_wait_warp(bar(B_S_FULL), (c - 1) & 1, abort_flag, p.err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tSB = tmem + lane_field + TM_SB + (c & 1) * (DK / 2);
            for (int g = 0; g < DK / 32; g++) {
                uint32_t r[32];
                tmem_ld32(tS + g * 32, r);
                tmem_wait_ld();
                if (GATE) {
                    const float* gm = gamma + s * DK + g * 32;
#pragma unroll
                    for (int i = 0; i < 32; i++) r[i] = __float_as_uint(__uint_as_float(r[i]) * gm[i]);
                    tmem_st32(tS + g * 32, r);
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++)
                    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                tmem_st16(tSB + g * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_READY));
        }
        if (ok && N > 0) ok = mbar_wait_warp(bar(B_S_FULL), (N - 1) & 1, abort_flag, p.err);
        if (ok) {
            tc_fence_after();
            float* fs = p.final_state ? p.final_state + (long)bh * DK * dv + j0 + j : nullptr;
            for (int g = 0; g < DK / 32; g++) {
                uint32_t r[32];
                tmem_ld32(tS + g * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const int d = g * 32 + i;
                    if (j < jvalid) {
                        if (fs) fs[(long)d * dv] = __uint_as_float(r[i]);
                    } else if (norm && j == 64 && p.final_z) {
                        p.final_z[(long)bh * DK + d] = __uint_as_float(r[i]);
                    }
                }
            }
        }
    } else if (warp < W_P0) {
        // ============================================================ output
        const int j = threadIdx.x - W_OUT0 * 32;
        for (int c = 0; c < N; c++) {
            const int ob = c & 1;
            bool ok = mbar_wait_warp(bar(B_O_FULL + ob), (c >> 1) & 1, abort_flag, p.err);
            uint32_t r0[32], r1[32];
            float* dn = den + ob * C;
            if (ok) {
                tc_fence_after();
                const uint32_t tO = tmem + lane_field + TM_O + ob * 64;
                tmem_ld32(tO, r0);
                tmem_ld32(tO + 32, r1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_EMPTY + ob));
                if (norm && j == 64) {
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        dn[t] = __uint_as_float(r0[t]);
                        dn[t + 32] = __uint_as_float(r1[t]);
                    }
                }
            }
            if (norm) ok = bar_red_and(2, 128, ok);
            if (!ok) break;
            const int nval = min(C, L - c * C);
            if (j < jvalid && j < dv - j0) {
                const long base = ((long)bh * L + (long)c * C) * dv + j0 + j;
                if (p.out_f32) {
                    float* o = static_cast<float*>(p.out) + base;
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float x = __uint_as_float(r0[t]);
                        if (norm) x = x / dn[t];
                        if (t < nval) o[(long)t * dv] = x;
                    }
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float x = __uint_as_float(r1[t]);
                        if (norm) x = x / dn[t + 32];
                        if (t + 32 < nval) o[(long)(t + 32) * dv] = x;
                    }
                } else {
                    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + base;
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float x = __uint_as_float(r0[t]);
                        if (norm) x = x / dn[t];
                        if (t < nval) o[(long)t * dv] = __float2bfloat16_rn(x);
                    }
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float x = __uint_as_float(r1[t]);
                        if (norm) x = x / dn[t + 32];
                        if (t + 32 < nval) o[(long)(t + 32) * dv] = __float2bfloat16_rn(x);
                    }
                }
            }
        }
    } else if (warp < W_TMA) {
        // ============================================================ P = tril(A) -> bf16
        const int t = threadIdx.x - W_P0 * 32;  // token row 0..63 (TMEM lanes 0..63)
        for (int c = 0; c < N; c++) {
            const int ob = c & 1;
            if (!mbar_wait_warp(bar(B_A_FULL + ob), (c >> 1) & 1, abort_flag, p.err)) break;
            if (!mbar_wait_warp(bar(B_P_EMPTY + ob), ((c >> 1) & 1) ^ 1, abort_flag, p.err)) break;
            tc_fence_after();
            uint32_t r[2][32];
            const uint32_t tA = tmem + lane_field + TM_A + ob * 64;
            tmem_ld32(tA, r[0]);
            tmem_ld32(tA + 32, r[1]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_A_EMPTY + ob));
            uint8_t* P = sm + Ly::off_p + ob * Ly::PB;
#pragma unroll
            for (int k8 = 0; k8 < 8; k8++) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int i = k8 * 8 + e;
                    const float a = __uint_as_float(r[i >> 5][i & 31]);
                    x[e] = (i <= t) ? a : 0.f;
                }
                uint4 w;
                w.x = pack_bf16x2(x[0], x[1]);
                w.y = pack_bf16x2(x[2], x[3]);
                w.z = pack_bf16x2(x[4], x[5]);
                w.w = pack_bf16x2(x[6], x[7]);
                *reinterpret_cast<uint4*>(P + sw128_offset(t, k8 * 8)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + ob));
        }
    } else if (warp == W_TMA) {
        // ============================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            if (GATE) tma_prefetch_desc(&p.tm_la);
            for (int c = 0; c < N; c++) {
                const int row = c * C;
                if (GATE) {
                    const int l = c % NL;
                    if (!mbar_wait(bar(B_LA_EMPTY + l), ((c / NL) & 1) ^ 1, abort_flag, p.err)) break;
                    mbar_arrive_expect_tx(bar(B_LA_FULL + l), Ly::LAB);
                    tma_load_3d(sbase + Ly::off_la + l * Ly::LAB, &p.tm_la, bar(B_LA_FULL + l), 0, row, bh);
                }
                const int s = c % NS;
                if (!mbar_wait(bar(B_QK_EMPTY + s), ((c / NS) & 1) ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(bar(B_QK_FULL + s), 2 * Ly::QB);
                const uint32_t qdst = sbase + Ly::off_qk + s * Ly::STAGE_QK;
                for (int a = 0; a < DK / 64; a++) {
                    tma_load_3d(qdst + a * 8192, &p.tm_q, bar(B_QK_FULL + s), a * 64, row, bh);
                    tma_load_3d(qdst + Ly::QB + a * 8192, &p.tm_k, bar(B_QK_FULL + s), a * 64, row, bh);
                }
                const int v = c % NV;
                if (!mbar_wait(bar(B_V_EMPTY + v), ((c / NV) & 1) ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(bar(B_V_FULL + v), nvb * 8192);
                for (int blk = 0; blk < nvb; blk++)
                    tma_load_3d(sbase + Ly::off_v + v * Ly::VB + blk * 8192, &p.tm_v, bar(B_V_FULL + v),
                                j0 + blk * 64, row, bh);
                last_issued = c;
            }
        }
    } else {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idA = make_idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t idS = make_idesc_bf16(128, DK, 1, 1);
            constexpr uint32_t idOi = make_idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t idOa = make_idesc_bf16(128, 64, 1, 0);
            for (int c = 0; c < N; c++) {
                const int s = c % NS, v = c % NV, ob = c & 1;
                const uint32_t Qs = sbase + Ly::off_qk + s * Ly::STAGE_QK;
                const uint32_t Ks = Qs + Ly::QB;
                const uint32_t Vs = sbase + Ly::off_v + v * Ly::VB;
                const uint32_t Ps = sbase + Ly::off_p + ob * Ly::PB;
                if (!mbar_wait(bar(B_QK_GATED + s), (c / NS) & 1, abort_flag, p.err)) break;
                if (!mbar_wait(bar(B_A_EMPTY + ob), ((c >> 1) & 1) ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                // A = Qh Kh^T (rows 64..127 of the M=128 tile read past the Q tile and are ignored)
#pragma unroll
                for (int kk = 0; kk < DK / 16; kk++) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_ss(tmem + TM_A + ob * 64, make_sdesc(Qs + off, 16, 1024), make_sdesc(Ks + off, 16, 1024),
                           idA, kk > 0);
                }
                mma_commit(bar(B_A_FULL + ob));
                if (!mbar_wait(bar(B_V_FULL + v), (c / NV) & 1, abort_flag, p.err)) break;
                if (!mbar_wait(bar(B_S_READY), c & 1, abort_flag, p.err)) break;
                tc_fence_after();
                // S^T += V^T Kh
#pragma unroll
                for (int kk = 0; kk < C / 16; kk++)
                    mma_ss(tmem + TM_S, make_sdesc(Vs + kk * 2048, 8192, 1024), make_sdesc(Ks + kk * 2048, 8192, 1024),
                           idS, 1);
                mma_commit(bar(B_S_FULL));
                if (!mbar_wait(bar(B_O_EMPTY + ob), ((c >> 1) & 1) ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                // O^T = S'^T Qh^T  (A operand: bf16 copy of the decayed state in TMEM)
#pragma unroll
                for (int kk = 0; kk < DK / 16; kk++) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_ts(tmem + TM_O + ob * 64, tmem + TM_SB + ob * (DK / 2) + kk * 8,
                           make_sdesc(Qs + off, 16, 1024), idOi, kk > 0);
                }
                if (!mbar_wait(bar(B_P_FULL + ob), (c >> 1) & 1, abort_flag, p.err)) break;
                tc_fence_after();
                // O^T += V^T P^T
#pragma unroll
                for (int kk = 0; kk < C / 16; kk++)
                    mma_ss(tmem + TM_O + ob * 64, make_sdesc(Vs + kk * 2048, 8192, 1024),
                           make_sdesc(Ps + kk * 32, 16, 1024), idOa, 1);
                mma_commit(bar(B_O_FULL + ob));
                mma_commit(bar(B_P_EMPTY + ob));
                mma_commit(bar(B_V_EMPTY + v));
                mma_commit(bar(B_QK_EMPTY + s));
            }
            // drain: every issued tcgen05 op has finished before TMEM is released
            mma_commit(bar(B_DRAIN));
            volatile int no_abort = 0;  // the drain wait is not cut short by an earlier abort
            mbar_wait(bar(B_DRAIN), 0, &no_abort, p.err);
        }
    }

    // ---------------------------------------------------------------- teardown
    if (warp == W_TMA && lane == 0 && *abort_flag && last_issued >= 0) {
        // wait (bounded) for loads that may still be in flight
        volatile int no_abort = 0;
        for (int c = max(0, last_issued - NS + 1); c <= last_issued; c++) {
            mbar_wait(bar(B_QK_FULL + c % NS), (c / NS) & 1, &no_abort, p.err);
            mbar_wait(bar(B_V_FULL + c % NV), (c / NV) & 1, &no_abort, p.err);
            if (GATE) mbar_wait(bar(B_LA_FULL + c % NL), (c / NL) & 1, &no_abort, p.err);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

CUresult encode_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int d0, int d1, int d2,
                   int box0, int box1, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)d0 * esize, (cuuint64_t)d0 * d1 * esize};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int DK, bool GATE>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    if (encode_3d(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, DK, a.L, BH, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_3d(&p.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, DK, a.L, BH, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_3d(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, a.dv, a.L, BH, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (GATE && encode_3d(&p.tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.log_alpha, DK, a.L, BH, DK, C,
                          CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.init_state = a.init_state;
    p.init_z = a.init_z;
    p.out = a.out;
    p.final_state = a.final_state;
    p.final_z = a.final_z;
    p.err = a.err_word;
    p.L = a.L;
    p.dv = a.dv;
    p.nchunks = (a.L + C - 1) / C;
    p.ntile = (a.dv + DVT - 1) / DVT;
    p.flags = a.flags;
    p.out_f32 = a.out_dtype == GLA_DTYPE_F32;
    auto kern = gla_prefill_tc_kernel<DK, GATE>;
    const int smem = Layout<DK>::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long grid = (long)BH * p.ntile;
    kern<<<dim3((unsigned)grid), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
    if (a.in_dtype != GLA_DTYPE_BF16) return false;
    if (a.flags & GLA_FLAG_FORCE_SIMT) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv < 64 || a.dv % 64 != 0) return false;
    if ((a.flags & GLA_FLAG_NORMALIZE) && a.dv != 64) return false;
    if (a.L < 1) return false;
    const long grid = (long)a.B * a.H * ((a.dv + DVT - 1) / DVT);
    if (grid > INT_MAX) return false;
    return true;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
    const bool gate = a.log_alpha != nullptr;
    if (a.dk == 64) return gate ? launch_t<64, true>(a, s) : launch_t<64, false>(a, s);
    return gate ? launch_t<128, true>(a, s) : launch_t<128, false>(a, s);
}

}  // namespace gla
