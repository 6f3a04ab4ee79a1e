// gla_delta_tc.cu -- the delta rule in chunk form on the tensor cores
// (tcgen05 + TMEM + TMA), sm_103a.
//
// "linear-attention" blog, Delta attention and its Prefill section: the writes
// of a sequence solve one lower-triangular system.  Per token (gated form: the
// state decays first, "Gated Linear Attention", GLA Recurrent Form)
//   S <- Diag(alpha_t) S;  u_t = beta_t (v_t - S^T k_t);  S <- S + k_t u_t^T;  o_t = S^T q_t.
// Over a chunk of C = 64 tokens starting from S_0, with b_t the in-chunk
// inclusive cumsum of log alpha and b_C its last value, put
//   Kr_t = k_t e^{b_t - b_C},  Kh_i = k_i e^{b_C - b_i},  Qh_t = q_t e^{b_t - b_C},
//   S' = Diag(e^{b_C}) S_0,   A = Kr Kh^T  (A_ti = sum_d k_td k_id e^{b_td - b_id}).
// Unrolling the recurrence, the chunk's writes U solve the unit lower-triangular
// system (I + Diag(beta) tril_strict(A)) U = Diag(beta) (V - Kr S'), so with
// T = (I + Diag(beta) tril_strict(A))^{-1} and M = T Diag(beta):
//   U = M V',  V' = V - Kr S'
//   O = Qh S' + tril(Qh Kh^T) U            (inclusive diagonal)
//   S_C = S' + Kh^T U.
// Every product is a tcgen05 MMA on 128-byte-swizzled bf16 tiles; T is the
// inverse of a 64 x 64 unit lower-triangular matrix, computed in fp32 by blocked
// forward substitution (16 x 16 diagonal blocks, then the off-diagonal blocks
// level by level).  The state copy S' and the writes U enter their products as
// bf16 high and low parts (x = hi + lo to ~2^-17); V' is formed in fp32 and
// rounded once to bf16.  Kr S' needs only the gate and the state, so it runs
// while the triangular inverse is computed.
//
// One CTA per (batch, head), d_k = d_v = 128: 256 worker threads, thread (d, hf)
// owning key channel d (TMEM lane d) and half hf of the chunk's tokens / of the
// state's columns, run the phases in turn behind their own barrier, with bounded
// waits; one more warp's first thread issues each group of tensor-core products
// once the workers have signalled that its operands are in place, so that issuing
// never holds up a worker.  A chunk over which some channel decays by more than
// e^-64 is outside the factorisation's range: the head is marked (a NaN pattern
// in the first output element of each 64-column block) and the token-by-token
// kernel recomputes exactly the marked heads afterwards.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int C = 64, D = 128;
constexpr int kWork = 256;         // worker threads
constexpr int kThr = kWork + 32;   // and the MMA-issuing warp
constexpr int TB = C * D * 2;    // bf16 [64][128]: two 8 KB atoms
constexpr int LAB = C * D * 4;   // fp32 log alpha tile
constexpr int PB = C * C * 2;    // bf16 [64][64]: one atom
constexpr int SB2 = D * D * 2;   // bf16 [128][128]: two 16 KB atoms
constexpr int LDF = C + 4;       // row stride (floats) of the fp32 [64][64] tiles: a row per lane
                                 // (and 16-byte groups of 8 rows) fall in distinct banks
constexpr int FB = C * LDF * 4;  // fp32 [64][64], rows LDF floats apart
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kStrongLog = -64.f;

struct DeltaTcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_la, tm_out;
    const float* beta;
    const float* init_state;
    void* out;
    float* final_state;
    unsigned* err;
    unsigned long long wait_ns;
    int L, nchunks, gate, out_f32;
    int out_tma;  // bf16 output staged in shared memory and written by bulk-tensor stores
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint16_t f2bf(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ uint32_t tile_off(int row, int col, int atom) {
    return (col >> 6) * atom + sw128_offset(row, col & 63);
}
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk, int atom) {
    return sdesc_const(16, 1024) | ((tile + (kk >> 2) * atom + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk, int lbo) {
    return sdesc_const(lbo, 1024) | ((tile + kk * 2048) >> 4);
}
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(x0, x1);
    const float2 h = unpack_bf16x2(hi);
    lo = pack_bf16x2(x0 - h.x, x1 - h.y);
}

// smem: q->Qh | k->Kh | Kr (later U high) | v (later U low) | log alpha | S' high | S' low |
//       M | P_m | N, then -(M Kr) | T | beta | exchange | barriers
constexpr int S_Q = 0, S_K = TB, S_KR = 2 * TB, S_V = 3 * TB, S_LA = 4 * TB, S_SH = 4 * TB + LAB,
              S_SL = S_SH + SB2, S_M = S_SL + SB2, S_PM = S_M + PB, S_N = S_PM + PB, S_T = S_N + FB,
              S_BETA = S_T + FB, S_X = S_BETA + C * 4, S_BAR = S_X + 5 * D * 4;
constexpr int S_SMEM = S_BAR + 128 + 1024;
static_assert(S_SMEM <= 227 * 1024, "shared memory budget");
// TMEM: S 0..127, O^T 128..191; 256..383 holds in turn Kr S', U and dS (read by the next chunk's
// state update before its Kr S' is issued); A and P 384..511 (64 each)
constexpr uint32_t T_S = 0, T_O = 128, T_U = 256, T_DS = 256, T_A = 384, T_P = 448;

// Barrier over the worker threads (named barrier 1; the MMA-issuing warp takes no part), and
// the same with an AND over a flag.
__device__ __forceinline__ void wbar() { asm volatile("barrier.cta.sync 1, %0;" ::"n"(kWork) : "memory"); }
__device__ __forceinline__ bool wbar_and(bool x) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)x), "n"(kWork)
        : "memory");
    return r != 0;
}

// A bounded wait on an mbarrier phase by every worker; false for all of them if any gave up.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const DeltaTcParams& p) {
    const bool ok = mbar_wait(bar, parity, abort_flag, p.err, p.wait_ns);
    return wbar_and(ok);
}

__device__ __forceinline__ void load_tiles(const DeltaTcParams& p, uint32_t bar, uint32_t sb, int c, int bh) {
    mbar_arrive_expect_tx(bar, 3 * TB);
    const CUtensorMap* maps[3] = {&p.tm_q, &p.tm_k, &p.tm_v};
    const uint32_t dst[3] = {sb + S_Q, sb + S_K, sb + S_V};
    for (int m = 0; m < 3; m++) {
        tma_load_3d(dst[m], maps[m], bar, 0, c * C, bh);
        tma_load_3d(dst[m] + 8192, maps[m], bar, 64, c * C, bh);
    }
}

// T = (I + N)^{-1} for N strictly lower triangular (fp32 [64][64] in shared
// memory, rows LDF floats apart): 16 x 16 diagonal blocks by forward
// substitution (one thread per column), then the off-diagonal blocks level by
// level,
//   T_IJ = -T_II sum_{J <= K < I} N_IK T_KJ   (I > J),
// the sums held in N's unused upper blocks between the level's two barriers.
// Only T's lower part (to the block diagonal) is written.  Every worker thread
// takes part (the barriers span the workers).
__device__ __forceinline__ void unit_lower_inverse(float* N, float* T, int tid) {
    // diagonal blocks, one thread per column j: x = T[., j] by forward substitution with the
    // updates applied as each entry becomes final (entries above j stay 0 and add nothing)
    if (tid < C) {
        const int blk = tid >> 4, j = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int t = 0; t < 16; t++) x[t] = (t == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; i++)
#pragma unroll
            for (int t = i + 1; t < 16; t++) x[t] -= N[(o + t) * LDF + o + i] * x[i];
#pragma unroll
        for (int t = 0; t < 16; t++) T[(o + t) * LDF + o + j] = x[t];
    }
    wbar();
#pragma unroll
    for (int lvl = 1; lvl < 4; lvl++) {
        // Y_IJ = sum_{J <= K < I} N_IK T_KJ for the 4 - lvl blocks (I, J = I - lvl): one entry per
        // thread and block (four partial sums), kept in N's unused upper block (J, I)
        const int a = tid >> 4, b = tid & 15;
#pragma unroll
        for (int n = 0; n < 4 - lvl; n++) {
            const int I = n + lvl, J = n;
            float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int Kb = J; Kb < I; Kb++)
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    const float4 nv = *reinterpret_cast<const float4*>(N + (I * 16 + a) * LDF + Kb * 16 + 4 * c4);
                    const float* tc = T + (Kb * 16 + 4 * c4) * LDF + J * 16 + b;
                    y[0] += nv.x * tc[0];
                    y[1] += nv.y * tc[LDF];
                    y[2] += nv.z * tc[2 * LDF];
                    y[3] += nv.w * tc[3 * LDF];
                }
            N[(J * 16 + a) * LDF + I * 16 + b] = (y[0] + y[1]) + (y[2] + y[3]);
        }
        wbar();
        // T_IJ = -T_II Y_IJ
#pragma unroll
        for (int n = 0; n < 4 - lvl; n++) {
            const int I = n + lvl, J = n;
            float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                const float4 tv = *reinterpret_cast<const float4*>(T + (I * 16 + a) * LDF + I * 16 + 4 * c4);
                const float* nc = N + (J * 16 + 4 * c4) * LDF + I * 16 + b;
                z[0] += tv.x * nc[0];
                z[1] += tv.y * nc[LDF];
                z[2] += tv.z * nc[2 * LDF];
                z[3] += tv.w * nc[3 * LDF];
            }
            T[(I * 16 + a) * LDF + J * 16 + b] = -((z[0] + z[1]) + (z[2] + z[3]));
        }
        wbar();
    }
}

__global__ void __launch_bounds__(kThr, 1) gla_delta_tc_kernel(const __grid_constant__ DeltaTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, d = tid & (D - 1), hf = tid >> 7;
    const int bh = blockIdx.x;
    const int L = p.L, N = p.nchunks;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    const uint32_t bar_t = smem_u32(&bars[0]), bar_l = smem_u32(&bars[1]), bar_mma = smem_u32(&bars[2]),
                   bar_drain = smem_u32(&bars[3]), bar_x = smem_u32(&bars[4]);
    // the workers' signals to the issuing thread: operands of A and P (h1), of Kr S' and the
    // state's share of O (h2), of U (h3), and of the rest of O and dS (h4)
    const uint32_t bar_h1 = smem_u32(&bars[5]), bar_h2 = smem_u32(&bars[6]), bar_h3 = smem_u32(&bars[7]),
                   bar_h4 = smem_u32(&bars[8]);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S_BAR + 96);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S_BAR + 100);
    float* xch = reinterpret_cast<float*>(sm + S_X);
    float* betas = reinterpret_cast<float*>(sm + S_BETA);
    float* Nf = reinterpret_cast<float*>(sm + S_N);
    float* Tf = reinterpret_cast<float*>(sm + S_T);
    int tiles_issued = 0, tiles_done = 0, la_issued = 0, la_done = 0;
    if (tid == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_l, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_h1, 1);
        mbar_init(bar_h2, 1);
        mbar_init(bar_h3, 1);
        mbar_init(bar_h4, 1);
        *abort_flag = 0;
        mbar_fence_init();
        load_tiles(p, bar_t, sb, 0, bh);
        tiles_issued++;
        if (p.gate) {
            mbar_arrive_expect_tx(bar_l, LAB);
            tma_load_3d(sb + S_LA, &p.tm_la, bar_l, 0, 0, bh);
            la_issued++;
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    if (tid < kWork) {
        const float* s0 = p.init_state ? p.init_state + ((long)bh * D + d) * D : nullptr;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e++) r[e] = __float_as_uint(s0 ? s0[h * 32 + e] : 0.f);
            tmem_st32(lane + T_S + h * 32, r);
        }
        tmem_wait_st();
    }
    const float* la = reinterpret_cast<const float*>(sm + S_LA);
    bool ok = true, strong = false;
    int mph = 0;  // phases of bar_mma completed
    float beta_next = (tid < C && tid < L) ? p.beta[(long)bh * L + tid] : 0.f;
    if (tid < kWork) {
        // the workers
        for (int c = 0; c < N; c++) {
            // log alpha was loaded during the previous chunk; q, k and v are waited for after the
            // gate's sums, which need log alpha alone
            if (p.gate) {
                if (!(ok = wait_all(bar_l, c & 1, abort_flag, p))) break;
                if (tid == 0) la_done++;
            }
            const int nval = min(C, L - c * C);
            // beta of this chunk (loaded one chunk ahead), and the next chunk's load in flight
            if (tid < C) {
                betas[tid] = beta_next;
                const int nn = min(C, L - (c + 1) * C);
                beta_next = (c + 1 < N && tid < nn) ? p.beta[(long)bh * L + (long)(c + 1) * C + tid] : 0.f;
            }
            // gate and factors: Kr = k e^{b_t - b_C} (new tile), Kh = k e^{b_C - b_t} and
            // Qh = q e^{b_t - b_C} in place.  Thread (channel pair gp, token quarter gq) takes
            // channels 2gp, 2gp + 1 over tokens 16 gq .. 16 gq + 15 (packed pairs); the quarter
            // sums of log alpha are exchanged for each quarter's prefix and the chunk total b_C.
            {
                const int gp = tid & 63, gq = tid >> 6, ch = 2 * gp;
                float2 b2 = make_float2(0.f, 0.f), bc2 = b2;
                float2 lx[16];  // this thread's log alpha pairs, read once for both passes
                if (p.gate) {
                    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 16; u++) {
                        lx[u] = *reinterpret_cast<const float2*>(la + (16 * gq + u) * D + ch);
                        s2.x += lx[u].x;
                        s2.y += lx[u].y;
                    }
                    *reinterpret_cast<float2*>(xch + gq * D + ch) = s2;
                    wbar();
#pragma unroll
                    for (int g = 0; g < 4; g++) {
                        const float2 u = *reinterpret_cast<const float2*>(xch + g * D + ch);
                        if (g < gq) {
                            b2.x += u.x;
                            b2.y += u.y;
                        }
                        bc2.x += u.x;
                        bc2.y += u.y;
                    }
                    if (gq == 0) *reinterpret_cast<float2*>(xch + 4 * D + ch) = bc2;  // b_C per channel
                    strong |= fminf(bc2.x, bc2.y) < kStrongLog;
                }
                if (!(ok = wait_all(bar_t, c & 1, abort_flag, p))) break;
                if (tid == 0) tiles_done++;
#pragma unroll
                for (int u = 0; u < 16; u++) {
                    const int t = 16 * gq + u;
                    const uint32_t o = tile_off(t, ch, 8192);
                    uint32_t* eq = reinterpret_cast<uint32_t*>(sm + S_Q + o);
                    uint32_t* ek = reinterpret_cast<uint32_t*>(sm + S_K + o);
                    uint32_t* er = reinterpret_cast<uint32_t*>(sm + S_KR + o);
                    const uint32_t kv = *ek;
                    if (p.gate) {
                        b2.x += lx[u].x;
                        b2.y += lx[u].y;
                        const float u0 = (b2.x - bc2.x) * kLog2e, u1 = (b2.y - bc2.y) * kLog2e;
                        const float fu0 = ex2f(u0), fu1 = ex2f(u1), fd0 = ex2f(-u0), fd1 = ex2f(-u1);
                        const float2 qf = unpack_bf16x2(*eq), kf = unpack_bf16x2(kv);
                        *eq = pack_bf16x2(qf.x * fu0, qf.y * fu1);
                        *er = pack_bf16x2(kf.x * fu0, kf.y * fu1);
                        *ek = pack_bf16x2(kf.x * fd0, kf.y * fd1);
                    } else {
                        *er = kv;
                    }
                }
            }
            fence_proxy_async_smem();  // the factors, read by the products below
            tc_fence_before();
            wbar();
            tc_fence_after();
            // b_C of this thread's key channel d, for the decay of the state below
            const float bC = p.gate ? xch[4 * D + d] : 0.f;
            if (tid == 0) {
                // log alpha is read until here: the next chunk's may load
                if (p.gate && c + 1 < N) {
                    mbar_arrive_expect_tx(bar_l, LAB);
                    tma_load_3d(sb + S_LA, &p.tm_la, bar_l, 0, (c + 1) * C, bh);
                    la_issued++;
                }
                mbar_arrive(bar_h1);  // A and P may be issued
                // the previous chunk's output staging (N's buffer) has been read by its stores
                if (p.out_tma) bulk_wait_group_read0();
            }
            // S' = e^{b_C} S, where S = S' + dS of the previous chunk (its state update is done here):
            // fp32 in TMEM, bf16 high and low copies in shared memory ([d][j], MN-major operand)
            {
                const float g = p.gate ? ex2f(bC * kLog2e) : 1.f;
#pragma unroll 1
                for (int h = 2 * hf; h < 2 * hf + 2; h++) {
                    uint32_t r[32];
                    tmem_ld32(lane + T_S + h * 32, r);
                    if (c > 0) {
                        uint32_t rd[32];
                        tmem_ld32(lane + T_DS + h * 32, rd);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; e++)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(rd[e]));
                    } else {
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int e8 = 0; e8 < 4; e8++) {
                        uint4 wh, wl;
                        const float* x = reinterpret_cast<const float*>(r + e8 * 8);
                        split_pair(x[0] * g, x[1] * g, wh.x, wl.x);
                        split_pair(x[2] * g, x[3] * g, wh.y, wl.y);
                        split_pair(x[4] * g, x[5] * g, wh.z, wl.z);
                        split_pair(x[6] * g, x[7] * g, wh.w, wl.w);
                        const uint32_t o = tile_off(d, h * 32 + e8 * 8, 16384);
                        *reinterpret_cast<uint4*>(sm + S_SH + o) = wh;
                        *reinterpret_cast<uint4*>(sm + S_SL + o) = wl;
                        // keep the fp32 S' for the state update
                        r[e8 * 8 + 0] = __float_as_uint(x[0] * g);
                        r[e8 * 8 + 1] = __float_as_uint(x[1] * g);
                        r[e8 * 8 + 2] = __float_as_uint(x[2] * g);
                        r[e8 * 8 + 3] = __float_as_uint(x[3] * g);
                        r[e8 * 8 + 4] = __float_as_uint(x[4] * g);
                        r[e8 * 8 + 5] = __float_as_uint(x[5] * g);
                        r[e8 * 8 + 6] = __float_as_uint(x[6] * g);
                        r[e8 * 8 + 7] = __float_as_uint(x[7] * g);
                    }
                    tmem_st32(lane + T_S + h * 32, r);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();  // S' high and low copies, read by the products after this barrier
            tc_fence_before();
            if (!(ok = wait_all(bar_mma, mph++ & 1, abort_flag, p))) break;
            tc_fence_after();
            if (tid == 0) mbar_arrive(bar_h2);
            // N = Diag(beta) tril_strict(A) in fp32; P_m = tril(P) in bf16 (rows t = lanes 0..63)
            if (d < C) {
                const int t = d;
                uint32_t ra[32], rp[32];
                tmem_ld32(lane + T_A + hf * 32, ra);
                tmem_ld32(lane + T_P + hf * 32, rp);
                tmem_wait_ld();
                const float bt = betas[t];
#pragma unroll
                for (int k8 = 0; k8 < 4; k8++) {
                    float x[8], n[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int i = hf * 32 + k8 * 8 + e;
                        x[e] = (i <= t) ? __uint_as_float(rp[k8 * 8 + e]) : 0.f;
                        n[e] = (i < t) ? bt * __uint_as_float(ra[k8 * 8 + e]) : 0.f;
                    }
                    float4* nr = reinterpret_cast<float4*>(Nf + t * LDF + hf * 32 + k8 * 8);
                    nr[0] = make_float4(n[0], n[1], n[2], n[3]);
                    nr[1] = make_float4(n[4], n[5], n[6], n[7]);
                    uint4 w;
                    w.x = pack_bf16x2(x[0], x[1]);
                    w.y = pack_bf16x2(x[2], x[3]);
                    w.z = pack_bf16x2(x[4], x[5]);
                    w.w = pack_bf16x2(x[6], x[7]);
                    *reinterpret_cast<uint4*>(sm + S_PM + sw128_offset(t, hf * 32 + k8 * 8)) = w;
                }
            }
            wbar();
            unit_lower_inverse(Nf, Tf, tid);
            if (!(ok = wait_all(bar_x, c & 1, abort_flag, p))) break;
            tc_fence_after();
            if (d >= C) {
                // M = T Diag(beta) in bf16 ([t][i], K-major operand); thread (t, half of the columns)
                const int t = d - C, h2 = hf;
#pragma unroll
                for (int k8 = 0; k8 < 4; k8++) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int i = h2 * 32 + k8 * 8 + e;
                        // T is unit lower triangular; its blocks above the block diagonal are not stored
                        x[e] = i <= t ? Tf[t * LDF + i] * betas[i] : 0.f;
                    }
                    uint4 w;
                    w.x = pack_bf16x2(x[0], x[1]);
                    w.y = pack_bf16x2(x[2], x[3]);
                    w.z = pack_bf16x2(x[4], x[5]);
                    w.w = pack_bf16x2(x[6], x[7]);
                    *reinterpret_cast<uint4*>(sm + S_M + sw128_offset(t, h2 * 32 + k8 * 8)) = w;
                }
            } else {
                // V' = V - X in bf16, in place over V ([t][j], MN-major operand; rows t = lanes 0..63)
                const int t = d;
#pragma unroll 1
                for (int h = 2 * hf; h < 2 * hf + 2; h++) {
                    uint32_t r[32];
                    tmem_ld32(lane + T_U + h * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k8 = 0; k8 < 4; k8++) {
                        uint4* pv = reinterpret_cast<uint4*>(sm + S_V + tile_off(t, h * 32 + k8 * 8, 8192));
                        const uint4 vv = *pv;
                        const float* x = reinterpret_cast<const float*>(r + k8 * 8);
                        const float2 v0 = unpack_bf16x2(vv.x), v1 = unpack_bf16x2(vv.y), v2 = unpack_bf16x2(vv.z),
                                     v3 = unpack_bf16x2(vv.w);
                        uint4 w;
                        w.x = pack_bf16x2(v0.x - x[0], v0.y - x[1]);
                        w.y = pack_bf16x2(v1.x - x[2], v1.y - x[3]);
                        w.z = pack_bf16x2(v2.x - x[4], v2.y - x[5]);
                        w.w = pack_bf16x2(v3.x - x[6], v3.y - x[7]);
                        *pv = w;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wbar();
            tc_fence_after();
            if (tid == 0) mbar_arrive(bar_h3);
            if (!(ok = wait_all(bar_mma, mph++ & 1, abort_flag, p))) break;
            tc_fence_after();
            // U in bf16 high and low parts over Kr and V ([i][j], MN-major operands; rows i = lanes 0..63)
            if (d < C) {
                const int i = d;
#pragma unroll 1
                for (int h = 2 * hf; h < 2 * hf + 2; h++) {
                    uint32_t r[32];
                    tmem_ld32(lane + T_U + h * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k8 = 0; k8 < 4; k8++) {
                        uint4 wh, wl;
                        const float* x = reinterpret_cast<const float*>(r + k8 * 8);
                        split_pair(x[0], x[1], wh.x, wl.x);
                        split_pair(x[2], x[3], wh.y, wl.y);
                        split_pair(x[4], x[5], wh.z, wl.z);
                        split_pair(x[6], x[7], wh.w, wl.w);
                        const uint32_t o = tile_off(i, h * 32 + k8 * 8, 8192);
                        *reinterpret_cast<uint4*>(sm + S_KR + o) = wh;
                        *reinterpret_cast<uint4*>(sm + S_V + o) = wl;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wbar();
            tc_fence_after();
            if (tid == 0) mbar_arrive(bar_h4);
            if (!(ok = wait_all(bar_mma, mph++ & 1, abort_flag, p))) break;
            tc_fence_after();
            // every product that reads this chunk's tiles has completed: load the next chunk's
            if (tid == 0 && c + 1 < N) {
                load_tiles(p, bar_t, sb, c + 1, bh);
                tiles_issued++;
            }
            // output: thread (j = d, half hf of the tokens) has o[t][j]; the state update
            // S = S' + dS is done with the next chunk's decay
            {
                uint32_t r[32];
                tmem_ld32(lane + T_O + hf * 32, r);
                tmem_wait_ld();
                if (p.out_tma) {
                    // bf16 into N's buffer (free after the inverse) as two row-major [64][64] boxes,
                    // written out below by two bulk-tensor stores (rows past L are clipped)
                    uint16_t* ob = reinterpret_cast<uint16_t*>(sm + S_N + (d >> 6) * 8192) + (hf * 32) * 64 + (d & 63);
#pragma unroll
                    for (int e = 0; e < 32; e++) ob[e * 64] = f2bf(__uint_as_float(r[e]));
                    fence_proxy_async_smem();
                } else {
                    const long row0 = (long)bh * L + (long)c * C + hf * 32;
#pragma unroll
                    for (int e = 0; e < 32; e++) {
                        if (hf * 32 + e < nval) {
                            const long idx = (row0 + e) * D + d;
                            if (p.out_f32)
                                static_cast<float*>(p.out)[idx] = __uint_as_float(r[e]);
                            else
                                static_cast<uint16_t*>(p.out)[idx] = f2bf(__uint_as_float(r[e]));
                        }
                    }
                }
            }
            tc_fence_before();
            wbar();
            if (p.out_tma && tid == 0) {
                tma_store_3d(&p.tm_out, sb + S_N, 0, c * C, bh);
                tma_store_3d(&p.tm_out, sb + S_N + 8192, 64, c * C, bh);
                bulk_commit_group();
            }
        }
    } else if (tid == kWork) {
        // the MMA-issuing thread: each group of products once the workers' signal says that its
        // operands are in place (their fences and barrier come before the signal)
        constexpr uint32_t id64 = make_idesc_bf16(128, 64, 0, 0), id128 = make_idesc_bf16(128, 128, 0, 1),
                           idO = make_idesc_bf16(128, 64, 1, 0), idS = make_idesc_bf16(128, 128, 1, 1);
        for (int c = 0; c < N; c++) {
            // A = Kr Kh^T and P = Qh Kh^T (M = 128: rows 64..127 read past the tile and are
            // ignored); they run while the workers decay and split the state
            if (!(ok = mbar_wait(bar_h1, c & 1, abort_flag, p.err, p.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_A, desc_k(sb + S_KR, kk, 8192), desc_k(sb + S_K, kk, 8192), id64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_P, desc_k(sb + S_Q, kk, 8192), desc_k(sb + S_K, kk, 8192), id64, kk > 0);
            mma_commit(bar_mma);
            // X = Kr S' (A = Kr K-major, B = S' high and low MN-major, N = 128; M = 128 as above),
            // then the state's share of the output, O^T = S'^T Qh^T (M = j: A = S' MN-major,
            // B = Qh K-major); both run during the triangular inverse
            if (!(ok = mbar_wait(bar_h2, c & 1, abort_flag, p.err, p.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_U, desc_k(sb + S_KR, kk, 8192), desc_mn(sb + S_SH, kk, 16384), id128, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_U, desc_k(sb + S_KR, kk, 8192), desc_mn(sb + S_SL, kk, 16384), id128, 1);
            mma_commit(bar_x);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_O, desc_mn(sb + S_SH, kk, 16384), desc_k(sb + S_Q, kk, 8192), idO, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++)
                mma_ss(tmem + T_O, desc_mn(sb + S_SL, kk, 16384), desc_k(sb + S_Q, kk, 8192), idO, 1);
            // U = M V' (A = M K-major, B = V' MN-major), N = 128
            if (!(ok = mbar_wait(bar_h3, c & 1, abort_flag, p.err, p.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + T_U, desc_k(sb + S_M, kk, 8192), desc_mn(sb + S_V, kk, 8192), id128, kk > 0);
            mma_commit(bar_mma);
            // O^T += U^T P_m^T (M = j: A = U MN-major, B = P_m K-major), then dS = Kh^T U
            // (A = Kh MN-major, B = U MN-major)
            if (!(ok = mbar_wait(bar_h4, c & 1, abort_flag, p.err, p.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + T_O, desc_mn(sb + S_KR, kk, 8192), desc_k(sb + S_PM, kk, 8192), idO, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + T_O, desc_mn(sb + S_V, kk, 8192), desc_k(sb + S_PM, kk, 8192), idO, 1);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + T_DS, desc_mn(sb + S_K, kk, 8192), desc_mn(sb + S_KR, kk, 8192), idS, kk > 0);
#pragma unroll
            for (int kk = 0; kk < C / 16; kk++)
                mma_ss(tmem + T_DS, desc_mn(sb + S_K, kk, 8192), desc_mn(sb + S_V, kk, 8192), idS, 1);
            mma_commit(bar_mma);
        }
    }
    if (p.out_tma && tid == 0) {
        // the stores have finished (shared memory stays valid, and the marks below come after them)
        bulk_wait_group0();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    if (tid == 0 && !ok) {
        // loads still in flight land before the CTA ends
        volatile int no_abort = 0;
        for (int n = tiles_done; n < tiles_issued; n++) mbar_wait(bar_t, n & 1, &no_abort, nullptr);
        for (int n = la_done; n < la_issued; n++) mbar_wait(bar_l, n & 1, &no_abort, nullptr);
    }
    if (tid == kWork) {
        // every product the issuing thread started has completed before TMEM is released
        volatile int no_abort = 0;
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, &no_abort, nullptr);
    }
    const bool mark = __syncthreads_or(strong) != 0;
    if (tid < kWork && ok && !mark && p.final_state) {
        // S = S' + dS of the last chunk (the initial state when there is none)
        float* fs = p.final_state + ((long)bh * D + d) * D;
#pragma unroll 1
        for (int h = 2 * hf; h < 2 * hf + 2; h++) {
            uint32_t r[32];
            tmem_ld32(lane + T_S + h * 32, r);
            if (N > 0) {
                uint32_t rd[32];
                tmem_ld32(lane + T_DS + h * 32, rd);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e++) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(rd[e]));
            } else {
                tmem_wait_ld();
            }
#pragma unroll
            for (int e = 0; e < 32; e++) fs[h * 32 + e] = __uint_as_float(r[e]);
        }
    }
    if (ok && mark && tid < D / 64) {
        // the token-by-token kernel recomputes this head: one mark per 64-column block
        const long idx = (long)bh * L * D + tid * 64;
        if (p.out_f32)
            static_cast<uint32_t*>(p.out)[idx] = kDeltaMarkF32;
        else
            static_cast<uint16_t*>(p.out)[idx] = kDeltaMarkBf16;
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

bool delta_tc_supported(const DeltaArgs& a) {
    return a.dk == D && a.dv == D && a.L >= 1 && !(a.flags & GLA_FLAG_FORCE_SIMT) &&
           (long)a.B * a.H <= 0x7fffffffL;
}

cudaError_t launch_delta_tc(const DeltaArgs& a, cudaStream_t s) {
    DeltaTcParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (encode(&p.tm_q, bf, 2, a.q, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS ||
        encode(&p.tm_k, bf, 2, a.k, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS ||
        encode(&p.tm_v, bf, 2, a.v, D, a.L, BH, 64, C, sw) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (a.log_alpha && encode(&p.tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.log_alpha, D, a.L, BH, D, C,
                              CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.beta = a.beta;
    p.init_state = a.init_state;
    p.out = a.out;
    p.final_state = a.final_state;
    p.err = a.err_word;
    p.wait_ns = a.wait_ns;
    p.L = a.L;
    p.nchunks = (a.L + C - 1) / C;
    p.gate = a.log_alpha != nullptr;
    p.out_f32 = a.out_dtype == GLA_DTYPE_F32;
    // bf16 output by bulk-tensor stores where the output allows a tensor map (16-byte aligned),
    // else by plain stores
    p.out_tma = !p.out_f32 && (reinterpret_cast<uintptr_t>(a.out) & 15) == 0 &&
                encode(&p.tm_out, bf, 2, a.out, D, a.L, BH, 64, C, CU_TENSOR_MAP_SWIZZLE_NONE) == CUDA_SUCCESS;
    cudaError_t e = cudaFuncSetAttribute(gla_delta_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S_SMEM);
    if (e != cudaSuccess) return e;
    gla_delta_tc_kernel<<<BH, kThr, S_SMEM, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // heads with a chunk outside the factorisation's range: the token-by-token kernel
    DeltaArgs r = a;
    r.only_marked = 1;
    return launch_delta(r, s);
}

}  // namespace gla
