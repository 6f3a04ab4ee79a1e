// gla_bwd_tc.cu -- backward pass of the gated recurrence in chunk form on the
// tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Method ("Gated Linear Attention", GLA Recurrent Form and Chunk-Wise
// Block-Parallel): the forward computes, per chunk of C = 64 tokens with b_t the
// in-chunk inclusive cumsum of log alpha and b_C its last value,
//   o_t = (q_t e^{b_t})^T S_{c-1} + sum_{i<=t} [sum_d q_td k_id e^{b_td - b_id}] v_i
//   S_c = Diag(e^{b_C}) S_{c-1} + sum_i (k_i e^{b_C - b_i}) v_i^T.
// With Qh_t = q_t e^{b_t - b_C}, Kh_i = k_i e^{b_C - b_i}, S' = Diag(e^{b_C}) S_{c-1},
// D = dO V^T and D_m / P_m = D / (Qh Kh^T) masked to i <= t, and G_c = dL/dS_c,
// differentiating those two lines gives, per chunk,
//   dq_t = e^{b_t - b_C} (S' do_t + (D_m Kh)_t)
//   dk_i = e^{b_C - b_i} (G_c v_i + (D_m^T Qh)_i)
//   dv_i = G_c^T Kh_i + (P_m^T dO)_i
//   G_{c-1} = Diag(e^{b_C}) (G_c + Qh^T dO)
// and the gate enters only through its cumulative sums, so
//   dlog_alpha_t = sum_{s >= t} (q_s dq_s - k_s dk_s)  (+ rowsum(dS_{L-1} S_{L-1}))
// -- the same identity the recurrent backward uses.
//
// Two kernels, one CTA of 256 threads per (batch, head): thread (d, hf) owns key
// channel d (tensor-memory lane d) and half hf of the chunk's tokens and of the
// state's columns (d_k = d_v = 128):
//   dq pass: chunks in order, S fp32 in TMEM; products D = dO V^T, dS = Kh^T V,
//            dQ^T = S'(TMEM) dO^T + Kh^T D_m^T; dq written with its factor.
//            At the end rowsum(dS_{L-1} S_{L-1}) is left in the last token's row
//            of dlog_alpha for the second pass.
//   dk/dv pass: chunks in reverse, G fp32 in TMEM; products P = Qh Kh^T,
//            D = dO V^T, dG = Qh^T dO, dK^T = G V^T + Qh^T D_m, dV^T = G^T Kh^T +
//            dO^T P_m; dk, dv, the gate gradient (suffix sums over the tokens,
//            reading q, k and the dq of the first pass) and dS_init.
// Every phase runs on all threads in turn (gate factors, products issued by one
// thread, epilogues), with bounded waits; the next chunk's tiles are loaded as
// soon as the last product that reads the current ones has completed, and its
// log alpha (two buffers) as soon as the current one has landed, so the copies
// overlap the work.  The state copies that enter the products (S' in
// the dq pass, G in the dk/dv pass) are split into bf16 high and low parts
// (x = hi + lo to about 2^-17), two products each: for slowly decaying gates the
// state carries most of a gradient, and one bf16 copy would set its error.  A chunk over which
// some channel decays by more than e^-64 is outside the factorisation's range;
// the dk/dv pass then marks the head (a NaN pattern in its dk and dv rows) and
// the recurrent kernel recomputes exactly the marked heads afterwards.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int C = 64;         // chunk length
constexpr int D = 128;        // d_k = d_v
constexpr int TB = C * D * 2;  // bf16 tile [64 tokens][128 channels]: two 8 KB swizzle atoms
constexpr int LAB = C * D * 4;  // fp32 log alpha tile
constexpr int PB = C * C * 2;  // bf16 [64][64] (one atom)
constexpr int GSB = D * D * 2;  // bf16 [128][128] state gradient copy: two 16 KB atoms
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kStrongLog = -64.f;

struct BwdTcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_la;
    const uint16_t* q;  // raw bf16 inputs (gate-gradient epilogue)
    const uint16_t* k;
    const float* init_state;
    const float* dfinal;
    float* dq;
    float* dk;
    float* dv;
    float* dla;
    float* dinit;
    unsigned* err;
    unsigned long long wait_ns;
    int L, nchunks, gate;
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint16_t f2bf(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Element (row, col) of a bf16 tile of rows of 128 channels stored as two 128-byte
// swizzled atoms of 64 columns, `atom` bytes apart.
__device__ __forceinline__ uint32_t tile_off(int row, int col, int atom) {
    return (col >> 6) * atom + sw128_offset(row, col & 63);
}

// Shared-memory descriptors (128-byte swizzle).  K-major: K steps of 16 elements
// (32 bytes) inside a 64-element atom row, `atom` bytes between the two atoms of
// a 128-wide K.  MN-major: K steps of 16 rows (2048 bytes), `lbo` bytes between
// the 64-element M/N blocks.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk, int atom) {
    return sdesc_const(16, 1024) | ((tile + (kk >> 2) * atom + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk, int lbo) {
    return sdesc_const(lbo, 1024) | ((tile + kk * 2048) >> 4);
}

// Bounded wait of every thread on an mbarrier phase; false (and the error record)
// when it runs out.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const BwdTcParams& p) {
    const bool ok = mbar_wait(bar, parity, abort_flag, p.err, p.wait_ns);
    return __syncthreads_and(ok) != 0;
}

// Loads of one chunk's bf16 tiles (two boxes of 64 channels each), and of its log alpha.
__device__ __forceinline__ void load_tiles(uint32_t bar, const CUtensorMap* const* maps, const uint32_t* dst, int n,
                                           int c, int bh) {
    mbar_arrive_expect_tx(bar, n * TB);
    for (int m = 0; m < n; m++) {
        tma_load_3d(dst[m], maps[m], bar, 0, c * C, bh);
        tma_load_3d(dst[m] + 8192, maps[m], bar, 64, c * C, bh);
    }
}
__device__ __forceinline__ void load_la(const BwdTcParams& p, uint32_t bar, uint32_t dst, int c, int bh) {
    mbar_arrive_expect_tx(bar, LAB);
    tma_load_3d(dst, &p.tm_la, bar, 0, c * C, bh);
}

// bf16 high and low parts of a pair: hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(x0, x1);
    const float2 h = unpack_bf16x2(hi);
    lo = pack_bf16x2(x0 - h.x, x1 - h.y);
}

// Columns [32 hf, 32 hf + 32) of rows 0..63 of a 64x64 fp32 accumulator in TMEM
// (row t = lane t), masked to i <= t, as bf16 into a [t][i] tile.  Warps whose
// lanes are 0..63.
__device__ __forceinline__ void mask_half(uint32_t taddr, uint8_t* dst, int t, int hf) {
    uint32_t r[32];
    tmem_ld32(taddr + hf * 32, r);
    tmem_wait_ld();
#pragma unroll
    for (int k8 = 0; k8 < 4; k8++) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = hf * 32 + k8 * 8 + e;
            x[e] = (i <= t) ? __uint_as_float(r[k8 * 8 + e]) : 0.f;
        }
        uint4 w;
        w.x = pack_bf16x2(x[0], x[1]);
        w.y = pack_bf16x2(x[2], x[3]);
        w.z = pack_bf16x2(x[4], x[5]);
        w.w = pack_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4*>(dst + sw128_offset(t, hf * 32 + k8 * 8)) = w;
    }
}

// Bulk copy of `bytes` contiguous bytes, global -> shared, completing on an mbarrier
// (both addresses 16-byte aligned, `bytes` a multiple of 16: the entry point checks the
// buffers' alignment and every row block here is a multiple of 256 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Loads issued by thread 0 and not yet waited for, so that a CTA that gives up
// waits for them before it leaves: tiles (one barrier) and log alpha (two).
struct Pending {
    int tiles_issued = 0, tiles_done = 0;
    int la_issued[2] = {0, 0}, la_done[2] = {0, 0};
    int epi_issued = 0, epi_done = 0;  // the dk/dv pass's epilogue rows (bar_e)
};

__device__ __forceinline__ void drain(const Pending& pn, uint32_t bar_t, const uint32_t* bar_l, uint32_t bar_drain,
                                      uint32_t bar_e = 0) {
    volatile int no_abort = 0;
    if (threadIdx.x == 0) {
        for (int n = pn.tiles_done; n < pn.tiles_issued; n++) mbar_wait(bar_t, n & 1, &no_abort, nullptr);
        for (int b = 0; b < 2; b++)
            for (int n = pn.la_done[b]; n < pn.la_issued[b]; n++) mbar_wait(bar_l[b], n & 1, &no_abort, nullptr);
        for (int n = pn.epi_done; n < pn.epi_issued; n++) mbar_wait(bar_e, n & 1, &no_abort, nullptr);
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, &no_abort, nullptr);
    }
    __syncthreads();
}

// Thread layout of both passes: 256 threads, thread (d, hf) = key channel d (TMEM lane d)
// and half hf of the chunk's tokens / of the state's 128 columns.
constexpr int kThr2 = 2 * D;

// ================================================================ dq pass
// smem: k | v | dO | log alpha x 2 | D_m | exchange | barriers
constexpr int A_K = 0, A_V = TB, A_DO = 2 * TB, A_LA = 3 * TB, A_DM = 3 * TB + 2 * LAB, A_X = A_DM + PB,
              A_BAR = A_X + 6 * D * 4;
constexpr int A_SMEM = A_BAR + 64 + 1024;
// TMEM: S 0..127, dS 128..255, bf16 S' high 256..319, D 320..383, dQ^T 384..447, S' low 448..511
constexpr uint32_t TA_S = 0, TA_DS = 128, TA_SB = 256, TA_D = 320, TA_Q = 384, TA_SL = 448;

__global__ void __launch_bounds__(kThr2, 1) gla_bwd_dq_kernel(const __grid_constant__ BwdTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, d = tid & (D - 1), hf = tid >> 7;
    const int bh = blockIdx.x;
    const int L = p.L, N = p.nchunks;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + A_BAR);
    const uint32_t bar_t = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]), bar_drain = smem_u32(&bars[2]);
    const uint32_t bar_l[2] = {smem_u32(&bars[3]), smem_u32(&bars[4])};
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + A_BAR + 48);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + A_BAR + 52);
    float* xch = reinterpret_cast<float*>(sm + A_X);  // [6][D]: quarter sums of log alpha, b_C, first-half sum
    const CUtensorMap* maps[3] = {&p.tm_k, &p.tm_v, &p.tm_do};
    const uint32_t dsts[3] = {sb + A_K, sb + A_V, sb + A_DO};
    Pending pn;
    if (tid == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_l[0], 1);
        mbar_init(bar_l[1], 1);
        *abort_flag = 0;
        mbar_fence_init();
        if (N > 0) {
            load_tiles(bar_t, maps, dsts, 3, 0, bh);
            pn.tiles_issued++;
            if (p.gate) {
                load_la(p, bar_l[0], sb + A_LA, 0, bh);
                pn.la_issued[0]++;
            }
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // lanes of this warp's quarter
    // S_{-1}: columns [64 hf, 64 hf + 64) of row d of the initial state
    {
        const float* s0 = p.init_state ? p.init_state + ((long)bh * D + d) * D : nullptr;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e++) r[e] = __float_as_uint(s0 ? s0[h * 32 + e] : 0.f);
            tmem_st32(lane + TA_S + h * 32, r);
        }
        tmem_wait_st();
    }
    bool ok = true;
    int c = 0;
    for (; c < N; c++) {
        const float* la = reinterpret_cast<const float*>(sm + A_LA + (c & 1) * LAB);
        // log alpha was loaded a chunk ahead; the tiles are waited for after the gate's sums
        if (p.gate) {
            if (!(ok = wait_all(bar_l[c & 1], (c >> 1) & 1, abort_flag, p))) break;
            if (tid == 0) {
                pn.la_done[c & 1]++;
                // the other buffer was last read in the previous chunk
                if (c + 1 < N) {
                    load_la(p, bar_l[(c + 1) & 1], sb + A_LA + ((c + 1) & 1) * LAB, c + 1, bh);
                    pn.la_issued[(c + 1) & 1]++;
                }
            }
        }
        const int nval = min(C, L - c * C);
        // the tiles, then D = dO V^T (M = 128, rows 64..127 read past the dO tile and are
        // ignored): it needs no gate factor, so it runs while the gate forms its factors
        auto tiles_then_d = [&]() -> bool {
            if (!wait_all(bar_t, c & 1, abort_flag, p)) return false;
            if (tid == 0) {
                pn.tiles_done++;
                tc_fence_after();
                constexpr uint32_t idD = make_idesc_bf16(128, 64, 0, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tmem + TA_D, desc_k(sb + A_DO, kk, 8192), desc_k(sb + A_V, kk, 8192), idD, kk > 0);
            }
            return true;
        };
        // gate: Kh = k e^{b_C - b_t} in place.  Thread (channel pair gp, token quarter gq) takes
        // channels 2gp, 2gp + 1 over tokens 16 gq .. 16 gq + 15 (packed pairs); the quarter sums
        // give each quarter's prefix, b_C and the first half's sum (the epilogue's start)
        if (p.gate) {
            const int gp = tid & 63, gq = tid >> 6, ch = 2 * gp;
            float2 s2 = make_float2(0.f, 0.f);
            float2 lx[16];  // this thread's log alpha pairs, read once for both passes
#pragma unroll
            for (int u = 0; u < 16; u++) {
                lx[u] = *reinterpret_cast<const float2*>(la + (16 * gq + u) * D + ch);
                s2.x += lx[u].x;
                s2.y += lx[u].y;
            }
            *reinterpret_cast<float2*>(xch + gq * D + ch) = s2;
            __syncthreads();
            float2 b2 = make_float2(0.f, 0.f), bc2 = b2;
            float2 q[4];
#pragma unroll
            for (int g = 0; g < 4; g++) {
                q[g] = *reinterpret_cast<const float2*>(xch + g * D + ch);
                if (g < gq) {
                    b2.x += q[g].x;
                    b2.y += q[g].y;
                }
                bc2.x += q[g].x;
                bc2.y += q[g].y;
            }
            if (gq == 0) {
                *reinterpret_cast<float2*>(xch + 4 * D + ch) = bc2;
                *reinterpret_cast<float2*>(xch + 5 * D + ch) = make_float2(q[0].x + q[1].x, q[0].y + q[1].y);
            }
            if (!(ok = tiles_then_d())) break;
            uint8_t* kt = sm + A_K;
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int t = 16 * gq + u;
                b2.x += lx[u].x;
                b2.y += lx[u].y;
                uint32_t* e = reinterpret_cast<uint32_t*>(kt + tile_off(t, ch, 8192));
                const float2 kf = unpack_bf16x2(*e);
                *e = pack_bf16x2(kf.x * ex2f((bc2.x - b2.x) * kLog2e), kf.y * ex2f((bc2.y - b2.y) * kLog2e));
            }
        }
        if (!p.gate && !(ok = tiles_then_d())) break;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // b_C of key channel d and the log-gate sum before this thread's half of the tokens
        const float bC = p.gate ? xch[4 * D + d] : 0.f, pre = (p.gate && hf) ? xch[5 * D + d] : 0.f;
        if (tid == 0) {
            // dS = Kh^T V (both MN-major)
            constexpr uint32_t idS = make_idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + TA_DS, desc_mn(sb + A_K, kk, 8192), desc_mn(sb + A_V, kk, 8192), idS, kk > 0);
            mma_commit(bar_mma);
        }
        if (!(ok = wait_all(bar_mma, 0, abort_flag, p))) break;
        tc_fence_after();
        // state, columns [64 hf, 64 hf + 64): S' = e^{b_C} S (bf16 high and low copies for the
        // dQ product), S = S' + dS
        {
            const float g = p.gate ? ex2f(bC * kLog2e) : 1.f;
#pragma unroll 1
            for (int h = 2 * hf; h < 2 * hf + 2; h++) {
                uint32_t rs[32], rd[32], pk[16], pl[16];
                tmem_ld32(lane + TA_S + h * 32, rs);
                tmem_ld32(lane + TA_DS + h * 32, rd);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float a0 = __uint_as_float(rs[e]) * g, a1 = __uint_as_float(rs[e + 1]) * g;
                    split_pair(a0, a1, pk[e / 2], pl[e / 2]);
                    rs[e] = __float_as_uint(a0 + __uint_as_float(rd[e]));
                    rs[e + 1] = __float_as_uint(a1 + __uint_as_float(rd[e + 1]));
                }
                tmem_st32(lane + TA_S + h * 32, rs);
                tmem_st16(lane + TA_SB + h * 16, pk);
                tmem_st16(lane + TA_SL + h * 16, pl);
            }
        }
        if (d < C) mask_half(lane + TA_D, sm + A_DM, d, hf);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            // dQ^T = (S'_hi + S'_lo) dO^T (A operands from TMEM) + Kh^T D_m^T
            constexpr uint32_t idQ = make_idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ts(tmem + TA_Q, tmem + TA_SB + kk * 8, desc_k(sb + A_DO, kk, 8192), idQ, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ts(tmem + TA_Q, tmem + TA_SL + kk * 8, desc_k(sb + A_DO, kk, 8192), idQ, 1);
            constexpr uint32_t idQ2 = make_idesc_bf16(128, 64, 1, 0);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + TA_Q, desc_mn(sb + A_K, kk, 8192), desc_k(sb + A_DM, kk, 8192), idQ2, 1);
            mma_commit(bar_mma);
        }
        if (!(ok = wait_all(bar_mma, 1, abort_flag, p))) break;
        tc_fence_after();
        // every product that reads this chunk's tiles has completed: load the next chunk's
        if (tid == 0 && c + 1 < N) {
            load_tiles(bar_t, maps, dsts, 3, c + 1, bh);
            pn.tiles_issued++;
        }
        // dq_t = e^{b_t - b_C} dQ^T[d][t] for this half's tokens
        {
            float* dqp = p.dq + ((long)bh * L + (long)c * C) * D + d;
            float b = pre;
            uint32_t r[32];
            tmem_ld32(lane + TA_Q + hf * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e++) {
                const int t = hf * 32 + e;
                float f = 1.f;
                if (p.gate) {
                    b += la[t * D + d];
                    f = ex2f((b - bC) * kLog2e);
                }
                if (t < nval) dqp[(long)t * D] = __uint_as_float(r[e]) * f;
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (!ok) {
        drain(pn, bar_t, bar_l, bar_drain);
    } else if (p.dla && p.dfinal) {
        // the final-state part of the gate gradient, rowsum(dS_{L-1} * S_{L-1}), for the second pass
        const float* df = p.dfinal + ((long)bh * D + d) * D;
        float s = 0.f;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
            tmem_ld32(lane + TA_S + h * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e++) s = fmaf(df[h * 32 + e], __uint_as_float(r[e]), s);
        }
        xch[hf * D + d] = s;
        __syncthreads();
        if (hf == 0) p.dla[((long)bh * L + L - 1) * D + d] = xch[d] + xch[D + d];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================================================ dk / dv pass
// smem: q | k | v | dO | log alpha x 2 | G high (bf16) | G low | P_m | D_m | exchange | barriers
constexpr int B_Q = 0, B_K = TB, B_V = 2 * TB, B_DO = 3 * TB, B_LA = 4 * TB, B_GS = 4 * TB + 2 * LAB,
              B_GL = B_GS + GSB, B_PM = B_GL + GSB, B_DM = B_PM + PB, B_X = B_DM + PB, B_BAR = B_X + 6 * D * 4;
constexpr int B_SMEM = B_BAR + 64 + 1024;
// TMEM: G 0..127, dG 128..255, P 256..319, D 320..383, dK^T 384..447, dV^T 448..511
constexpr uint32_t TB_G = 0, TB_DG = 128, TB_P = 256, TB_D = 320, TB_K = 384, TB_V = 448;

__global__ void __launch_bounds__(kThr2, 1) gla_bwd_dkdv_kernel(const __grid_constant__ BwdTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, d = tid & (D - 1), hf = tid >> 7;
    const int bh = blockIdx.x;
    const int L = p.L, N = p.nchunks;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + B_BAR);
    const uint32_t bar_t = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]), bar_drain = smem_u32(&bars[2]);
    const uint32_t bar_l[2] = {smem_u32(&bars[3]), smem_u32(&bars[4])};
    const uint32_t bar_e = smem_u32(&bars[5]);  // the epilogue's rows of q, k and dq
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + B_BAR + 48);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + B_BAR + 52);
    float* xch = reinterpret_cast<float*>(sm + B_X);  // [6][D]: gate quarter sums, b_C, second-half sum
    const CUtensorMap* maps[4] = {&p.tm_q, &p.tm_k, &p.tm_v, &p.tm_do};
    const uint32_t dsts[4] = {sb + B_Q, sb + B_K, sb + B_V, sb + B_DO};
    Pending pn;
    if (tid == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_l[0], 1);
        mbar_init(bar_l[1], 1);
        mbar_init(bar_e, 1);
        *abort_flag = 0;
        mbar_fence_init();
        if (N > 0) {
            load_tiles(bar_t, maps, dsts, 4, N - 1, bh);
            pn.tiles_issued++;
            if (p.gate) {
                load_la(p, bar_l[0], sb + B_LA, N - 1, bh);
                pn.la_issued[0]++;
            }
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    // G_{N-1} = dL/dS_{L-1}: columns [64 hf, 64 hf + 64) of row d of dfinal
    {
        const float* g0 = p.dfinal ? p.dfinal + ((long)bh * D + d) * D : nullptr;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e++) r[e] = __float_as_uint(g0 ? g0[h * 32 + e] : 0.f);
            tmem_st32(lane + TB_G + h * 32, r);
        }
        tmem_wait_st();
    }
    // running suffix of the gate gradient of channel d over the chunks done so far (starts from
    // the final-state part the dq pass left in the last token's row)
    float acc = 0.f;
    if (p.dla && p.dfinal) acc = p.dla[((long)bh * L + L - 1) * D + d];
    bool ok = true, strong = false;
    int it = 0;
    for (int c = N - 1; c >= 0; c--, it++) {
        const float* la = reinterpret_cast<const float*>(sm + B_LA + (it & 1) * LAB);
        // log alpha was loaded a chunk ahead; the tiles are waited for after the gate's sums
        if (p.gate) {
            if (!(ok = wait_all(bar_l[it & 1], (it >> 1) & 1, abort_flag, p))) break;
            if (tid == 0) {
                pn.la_done[it & 1]++;
                if (c > 0) {
                    load_la(p, bar_l[(it + 1) & 1], sb + B_LA + ((it + 1) & 1) * LAB, c - 1, bh);
                    pn.la_issued[(it + 1) & 1]++;
                }
            }
        }
        const int nval = min(C, L - c * C);
        // the epilogue reads this chunk's rows of q, k and dq: bring them into L2 now, while
        // the products run (they are copied to shared memory once the products are done)
        if (tid == 0 && p.dla) {
            const long row0 = (long)bh * L + (long)c * C;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.dq + row0 * D), "r"(nval * D * 4)
                         : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.q + row0 * D), "r"(nval * D * 2)
                         : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.k + row0 * D), "r"(nval * D * 2)
                         : "memory");
        }
        // gate: Qh = q e^{b_t - b_C}, Kh = k e^{b_C - b_t} in place.  Thread (channel pair gp,
        // token quarter gq) takes channels 2gp, 2gp + 1 over tokens 16 gq .. 16 gq + 15 (packed
        // pairs); the quarter sums of log alpha give each quarter's prefix, b_C and the sum over
        // the second half (tokens 32..63) that the epilogue starts from.
        if (p.gate) {
            const int gp = tid & 63, gq = tid >> 6, ch = 2 * gp;
            float2 s2 = make_float2(0.f, 0.f);
            float2 lx[16];  // this thread's log alpha pairs, read once for both passes
#pragma unroll
            for (int u = 0; u < 16; u++) {
                lx[u] = *reinterpret_cast<const float2*>(la + (16 * gq + u) * D + ch);
                s2.x += lx[u].x;
                s2.y += lx[u].y;
            }
            *reinterpret_cast<float2*>(xch + gq * D + ch) = s2;
            __syncthreads();
            float2 b2 = make_float2(0.f, 0.f), bc2 = b2;
            float2 q[4];
#pragma unroll
            for (int g = 0; g < 4; g++) {
                q[g] = *reinterpret_cast<const float2*>(xch + g * D + ch);
                if (g < gq) {
                    b2.x += q[g].x;
                    b2.y += q[g].y;
                }
                bc2.x += q[g].x;
                bc2.y += q[g].y;
            }
            if (gq == 0) {
                *reinterpret_cast<float2*>(xch + 4 * D + ch) = bc2;
                *reinterpret_cast<float2*>(xch + 5 * D + ch) = make_float2(q[2].x + q[3].x, q[2].y + q[3].y);
            }
            strong |= fminf(bc2.x, bc2.y) < kStrongLog;
            if (!(ok = wait_all(bar_t, it & 1, abort_flag, p))) break;
            if (tid == 0) pn.tiles_done++;
            uint8_t* qt = sm + B_Q;
            uint8_t* kt = sm + B_K;
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int t = 16 * gq + u;
                b2.x += lx[u].x;
                b2.y += lx[u].y;
                const uint32_t o = tile_off(t, ch, 8192);
                uint32_t* eq = reinterpret_cast<uint32_t*>(qt + o);
                uint32_t* ek = reinterpret_cast<uint32_t*>(kt + o);
                const float u0 = (b2.x - bc2.x) * kLog2e, u1 = (b2.y - bc2.y) * kLog2e;
                const float2 qf = unpack_bf16x2(*eq), kf = unpack_bf16x2(*ek);
                *eq = pack_bf16x2(qf.x * ex2f(u0), qf.y * ex2f(u1));
                *ek = pack_bf16x2(kf.x * ex2f(-u0), kf.y * ex2f(-u1));
            }
        }
        if (!p.gate) {
            if (!(ok = wait_all(bar_t, it & 1, abort_flag, p))) break;
            if (tid == 0) pn.tiles_done++;
        }
        fence_proxy_async_smem();  // the factors, read by the products below
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // b_C of key channel d (the state decay) and its sum of log alpha over tokens 32..63
        const float bC = p.gate ? xch[4 * D + d] : 0.f, part1 = p.gate ? xch[5 * D + d] : 0.f;
        if (tid == 0) {
            constexpr uint32_t id64 = make_idesc_bf16(128, 64, 0, 0);
            // P = Qh Kh^T and D = dO V^T (M = 128: rows 64..127 read past the tile and are ignored)
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_P, desc_k(sb + B_Q, kk, 8192), desc_k(sb + B_K, kk, 8192), id64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_D, desc_k(sb + B_DO, kk, 8192), desc_k(sb + B_V, kk, 8192), id64, kk > 0);
            // dG = Qh^T dO
            constexpr uint32_t id128 = make_idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + TB_DG, desc_mn(sb + B_Q, kk, 8192), desc_mn(sb + B_DO, kk, 8192), id128, kk > 0);
            mma_commit(bar_mma);
        }
        // bf16 high and low copies of G_c into shared memory: columns [64 hf, 64 hf + 64) of row d
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
            tmem_ld32(lane + TB_G + h * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 4; e8++) {
                uint4 wh, wl;
                const float* x = reinterpret_cast<const float*>(r + e8 * 8);
                split_pair(x[0], x[1], wh.x, wl.x);
                split_pair(x[2], x[3], wh.y, wl.y);
                split_pair(x[4], x[5], wh.z, wl.z);
                split_pair(x[6], x[7], wh.w, wl.w);
                const uint32_t o = tile_off(d, h * 32 + e8 * 8, 16384);
                *reinterpret_cast<uint4*>(sm + B_GS + o) = wh;
                *reinterpret_cast<uint4*>(sm + B_GL + o) = wl;
            }
        }
        fence_proxy_async_smem();  // G's high and low copies, read by the second product group
        tc_fence_before();
        if (!(ok = wait_all(bar_mma, 0, abort_flag, p))) break;
        tc_fence_after();
        if (d < C) {
            mask_half(lane + TB_P, sm + B_PM, d, hf);
            mask_half(lane + TB_D, sm + B_DM, d, hf);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            // dK^T = (G_hi + G_lo) V^T + Qh^T D_m
            constexpr uint32_t idK1 = make_idesc_bf16(128, 64, 0, 0), idK2 = make_idesc_bf16(128, 64, 1, 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_K, desc_k(sb + B_GS, kk, 16384), desc_k(sb + B_V, kk, 8192), idK1, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_K, desc_k(sb + B_GL, kk, 16384), desc_k(sb + B_V, kk, 8192), idK1, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + TB_K, desc_mn(sb + B_Q, kk, 8192), desc_mn(sb + B_DM, kk, 8192), idK2, 1);
            // dV^T = (G_hi + G_lo)^T Kh^T + dO^T P_m
            constexpr uint32_t idV1 = make_idesc_bf16(128, 64, 1, 0), idV2 = make_idesc_bf16(128, 64, 1, 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_V, desc_mn(sb + B_GS, kk, 16384), desc_k(sb + B_K, kk, 8192), idV1, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + TB_V, desc_mn(sb + B_GL, kk, 16384), desc_k(sb + B_K, kk, 8192), idV1, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + TB_V, desc_mn(sb + B_DO, kk, 8192), desc_mn(sb + B_PM, kk, 8192), idV2, 1);
            mma_commit(bar_mma);
        }
        if (!(ok = wait_all(bar_mma, 1, abort_flag, p))) break;
        tc_fence_after();
        // every product that reads this chunk's tiles has completed: load the next chunk's
        if (tid == 0 && c > 0) {
            load_tiles(bar_t, maps, dsts, 4, c - 1, bh);
            pn.tiles_issued++;
        }
        // epilogue for this half's tokens, last to first: dk_i = e^{b_C - b_i} dK^T[d][i],
        // dv_i = dV^T[j = d][i], and the gate gradient's suffix sums
        {
            const long row0 = (long)bh * L + (long)c * C;
            // the gate gradient needs this chunk's rows of q, k and dq: one bulk copy each into
            // the space of G's bf16 copies (free until the next chunk's split), while the dk and
            // dv stores go out
            uint16_t* qs = reinterpret_cast<uint16_t*>(sm + B_GS);
            uint16_t* ks = qs + C * D;
            float* dqs = reinterpret_cast<float*>(sm + B_GL);
            if (tid == 0 && p.dla) {
                mbar_arrive_expect_tx(bar_e, nval * D * 8);
                bulk_load(sb + B_GS, p.q + row0 * D, nval * D * 2, bar_e);
                bulk_load(sb + B_GS + C * D * 2, p.k + row0 * D, nval * D * 2, bar_e);
                bulk_load(sb + B_GL, p.dq + row0 * D, nval * D * 4, bar_e);
                pn.epi_issued++;
            }
            float* dkp = p.dk + row0 * D + d;
            float* dvp = p.dv + row0 * D + d;
            float r_suf = hf ? 0.f : part1;  // b_C - b_i: sum of log alpha over (i, C)
            float gl[32];                    // suffix of q dq - k dk inside this half
            float loc = 0.f;
            uint32_t rk[32], rv[32];
            tmem_ld32(lane + TB_K + hf * 32, rk);
            tmem_ld32(lane + TB_V + hf * 32, rv);
            tmem_wait_ld();
#pragma unroll
            for (int e = 31; e >= 0; e--) {
                const int i = hf * 32 + e;
                const float f = p.gate ? ex2f(r_suf * kLog2e) : 1.f;
                const float dki = __uint_as_float(rk[e]) * f;
                rk[e] = __float_as_uint(dki);
                if (i < nval) {
                    dkp[(long)i * D] = dki;
                    dvp[(long)i * D] = __uint_as_float(rv[e]);
                }
                if (p.gate) r_suf += la[i * D + d];
            }
            if (p.dla) {
                if (!(ok = wait_all(bar_e, it & 1, abort_flag, p))) break;
                if (tid == 0) pn.epi_done++;
#pragma unroll
                for (int e = 31; e >= 0; e--) {
                    const int i = hf * 32 + e;
                    gl[e] = 0.f;
                    if (i < nval) {
                        loc += bf2f(qs[i * D + d]) * dqs[i * D + d] - bf2f(ks[i * D + d]) * __uint_as_float(rk[e]);
                        gl[e] = loc;
                    }
                }
            }
            if (p.dla) {
                // tokens of the second half come after the first half's in the suffix sums
                __syncthreads();  // xch was last read by the gate of this chunk
                xch[hf * D + d] = loc;
                __syncthreads();
                const float off = acc + (hf ? 0.f : xch[D + d]);
                float* dlp = p.dla + row0 * D + d;
#pragma unroll
                for (int e = 0; e < 32; e++) {
                    const int i = hf * 32 + e;
                    if (i < nval) dlp[(long)i * D] = off + gl[e];
                }
                acc += xch[d] + xch[D + d];
            }
        }
        // G_{c-1} = e^{b_C} (G_c + dG), columns [64 hf, 64 hf + 64)
        {
            const float g = p.gate ? ex2f(bC * kLog2e) : 1.f;
#pragma unroll 1
            for (int h = 2 * hf; h < 2 * hf + 2; h++) {
                uint32_t rg[32], rd[32];
                tmem_ld32(lane + TB_G + h * 32, rg);
                tmem_ld32(lane + TB_DG + h * 32, rd);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e++)
                    rg[e] = __float_as_uint(g * (__uint_as_float(rg[e]) + __uint_as_float(rd[e])));
                tmem_st32(lane + TB_G + h * 32, rg);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
    }
    if (!ok) drain(pn, bar_t, bar_l, bar_drain, bar_e);
    const bool mark = __syncthreads_or(strong) != 0;
    if (ok && !mark && p.dinit) {
        float* di = p.dinit + ((long)bh * D + d) * D;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
            tmem_ld32(lane + TB_G + h * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e++) di[h * 32 + e] = __uint_as_float(r[e]);
        }
    }
    if (ok && mark && tid < D / 32) {
        // the exact recurrent backward recomputes this head: one mark per row and column block
        reinterpret_cast<uint32_t*>(p.dk)[(long)bh * L * D + tid * 32] = kBwdMark;
        reinterpret_cast<uint32_t*>(p.dv)[(long)bh * L * D + tid * 32] = kBwdMark;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

CUresult encode(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int d0, int d1, int d2,
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

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
    return a.in_dtype == GLA_DTYPE_BF16 && a.dk == D && a.dv == D && !(a.flags & GLA_FLAG_SCALAR_GATE) &&
           !(a.flags & GLA_FLAG_FORCE_SIMT) && a.L >= 1 && (long)a.B * a.H <= 0x7fffffffL;
}

cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
    BwdTcParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (encode(&p.tm_q, bf, 2, a.q, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS ||
        encode(&p.tm_k, bf, 2, a.k, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS ||
        encode(&p.tm_v, bf, 2, a.v, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS ||
        encode(&p.tm_do, bf, 2, a.dout, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (a.log_alpha && encode(&p.tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.log_alpha, D, a.L, BH, D, C,
                              CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.q = static_cast<const uint16_t*>(a.q);
    p.k = static_cast<const uint16_t*>(a.k);
    p.init_state = a.init_state;
    p.dfinal = a.dfinal;
    p.dq = a.dq;
    p.dk = a.dk_out;
    p.dv = a.dv_out;
    p.dla = a.dlog_alpha;
    p.dinit = a.dinit;
    p.err = a.err_word;
    p.wait_ns = a.wait_ns;
    p.L = a.L;
    p.nchunks = (a.L + C - 1) / C;
    p.gate = a.log_alpha != nullptr;
    cudaError_t e = cudaFuncSetAttribute(gla_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gla_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, B_SMEM);
    if (e != cudaSuccess) return e;
    gla_bwd_dq_kernel<<<BH, kThr2, A_SMEM, s>>>(p);
    gla_bwd_dkdv_kernel<<<BH, kThr2, B_SMEM, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // heads with a chunk outside the factorisation's range: the exact recurrent kernel
    BwdArgs r = a;
    r.only_marked = 1;
    return launch_bwd(r, s);
}

}  // namespace gla
