// gla_bwd.cu -- gradients of the gated recurrence, token by token.
//
// "Gated Linear Attention", GLA Recurrent Form:  S_t = Diag(alpha_t) S_{t-1} +
// k_t v_t^T,  o_t = S_t^T q_t.  Given dL/do_t (dout) and dL/dS_{L-1} (dfinal),
// reverse mode gives, with G_t = dL/dS_t (the total gradient reaching S_t),
//   G_t = Diag(alpha_{t+1}) G_{t+1} + q_t dout_t^T     (G_{L-1} = dfinal + q dout^T)
//   dq_t = S_t dout_t,  dk_t = G_t v_t,  dv_t = G_t^T k_t,
//   dS_{-1} = Diag(alpha_0) G_0.
// For the gate, write b_t = sum_{u <= t} log alpha_u (per channel): every
// pairing of a query q_t with a key k_i carries e^{b_t - b_i}, so
// dL/db_s = q_s * dq_s - k_s * dk_s (+ rowsum(dfinal * S_{L-1}) at s = L-1),
// and log alpha_t enters every b_s with s >= t:
//   dlog_alpha_t = sum_{s >= t} (q_s * dq_s - k_s * dk_s) + rowsum(dfinal * S_{L-1}).
// (The same chunk-form reading the forward uses: the gate's cumulative sums
// are the only place log alpha appears.)
//
// Two kinds of CTA share one launch:
//  * row CTAs own 64 key rows of one head, all value columns.  Rows evolve on
//    their own (S_t[i,:] needs alpha_t[i], k_t[i] and v_t), so a forward sweep
//    carries S and emits dq (a reduction over the value columns), and a
//    reverse sweep carries G and emits dk, the running gate sum and dS_{-1}.
//    Lane (cg, rp) of a warp holds rows warp*4 + 2 rp + {0, 1} as fp32 pairs
//    over the value columns [cg * CPL, (cg + 1) * CPL).
//  * column CTAs own 64 value columns: a reverse sweep carries G column-wise
//    and emits dv (a reduction over the key rows).  Lane (rg, cp) holds rows
//    [rg * RPL, (rg + 1) * RPL) of the column pair 2 cp.
// Reductions are four butterfly shuffles across the sixteen lane groups.
// Tokens are staged in shared memory 16 at a time, double buffered.  Row CTAs
// come first in the grid: they do two sweeps, the column CTAs one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTB = 16;            // tokens staged per round
constexpr int kBlock = 4 * kWarps; // rows per row CTA, columns per column CTA

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }

// sum over the sixteen lane groups (lane bits 1..4)
__device__ __forceinline__ float2 group_sum(float2 x) {
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, m);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, m);
    }
    return x;
}

template <typename T>
__device__ __forceinline__ float to_f(T x) {
    if constexpr (std::is_same<T, float>::value)
        return x;
    else
        return __bfloat162float(x);
}

// N consecutive floats of a staged group (16-byte aligned when N >= 4)
template <int N>
__device__ __forceinline__ void load_run(const float* p, float (&r)[N]) {
    if constexpr (N >= 4) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + i);
            r[i] = x.x, r[i + 1] = x.y, r[i + 2] = x.z, r[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float2 x = *reinterpret_cast<const float2*>(p + i);
            r[i] = x.x, r[i + 1] = x.y;
        }
    }
}

// Staging of one round of tokens.  "Wide" arrays span the full dimension that
// the CTA's lanes split in sixteen groups of W floats (padded to W + 4 per
// group); "narrow" arrays span only the CTA's own 64-entry block.
template <int W>
struct Stage {
    static constexpr int FULL = 16 * W;
    static constexpr int STRIDE = W + 4;
    static constexpr int ROW = 16 * STRIDE;
    __device__ static constexpr int pidx(int x) { return (x / W) * STRIDE + x % W; }
    static constexpr int NW = (kTB * FULL + kThreads - 1) / kThreads;    // wide loads per thread
    static constexpr int NN = (kTB * kBlock + kThreads - 1) / kThreads;  // narrow loads per thread
};

// ---- row CTAs: dq (forward sweep); dk, dlog_alpha, dS_{-1} (reverse sweep) ----
// Wide arrays are over the value columns (W = CPL): v, dout.  Narrow arrays over
// the CTA's 64 key rows: k, alpha, and q, dq in the reverse sweep.
template <int CPL, bool GATE, typename T>
__device__ __forceinline__ void rows_body(const BwdArgs& a, float* sm, int blk) {
    using St = Stage<CPL>;
    constexpr int DV = St::FULL;
    constexpr int BUF = kTB * (2 * St::ROW + 4 * kBlock);
    const int L = a.L, dk = a.dk;
    const long bh = blockIdx.x;
    const int row0 = blk * kBlock, nrows = min(kBlock, dk - row0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = lane >> 1, rp = lane & 1;
    const int rl = warp * 4 + rp * 2;  // this lane's first row within the block
    const bool active = warp * 4 < nrows;  // dk is a multiple of 4: a warp is all or nothing
    const int r = row0 + rl;

    const T* q = static_cast<const T*>(a.q) + bh * (long)L * dk;
    const T* k = static_cast<const T*>(a.k) + bh * (long)L * dk;
    const T* v = static_cast<const T*>(a.v) + bh * (long)L * DV;
    const T* dout = static_cast<const T*>(a.dout) + bh * (long)L * DV;
    const float* la = GATE ? a.log_alpha + bh * (long)L * dk : nullptr;
    float* dq = a.dq + bh * (long)L * dk;

    T rv[St::NW], rd[St::NW], rk[St::NN], rq[St::NN];
    float ra[St::NN], rdq[St::NN];
    // round [t0, t0 + n): global -> registers; REV also fetches q and dq
    auto fetch = [&](int t0, int n, bool rev) {
#pragma unroll
        for (int m = 0; m < St::NW; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DV) {
                const long g = (long)t0 * DV + idx;
                rv[m] = v[g];
                rd[m] = dout[g];
            }
        }
#pragma unroll
        for (int m = 0; m < St::NN; m++) {
            const int idx = tid + m * kThreads;
            const int t = idx / kBlock, i = idx % kBlock;
            if (t < n && i < nrows) {
                const long g = (long)(t0 + t) * dk + row0 + i;
                rk[m] = k[g];
                if (GATE) ra[m] = la[g];
                if (rev) {
                    rq[m] = q[g];
                    if (GATE) rdq[m] = dq[g];
                }
            }
        }
    };
    auto stage = [&](int n, bool rev, float* buf) {
        float* s_v = buf;
        float* s_d = s_v + kTB * St::ROW;
        float* s_k = s_d + kTB * St::ROW;
        float* s_a = s_k + kTB * kBlock;
        float* s_q = s_a + kTB * kBlock;
        float* s_dq = s_q + kTB * kBlock;
#pragma unroll
        for (int m = 0; m < St::NW; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DV) {
                const int o = (idx / DV) * St::ROW + St::pidx(idx % DV);
                s_v[o] = to_f(rv[m]);
                s_d[o] = to_f(rd[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < St::NN; m++) {
            const int idx = tid + m * kThreads;
            if (idx / kBlock < n && idx % kBlock < nrows) {
                s_k[idx] = to_f(rk[m]);
                s_a[idx] = GATE ? __expf(ra[m]) : 1.f;
                if (rev) {
                    s_q[idx] = to_f(rq[m]);
                    s_dq[idx] = GATE ? rdq[m] : 0.f;
                }
            }
        }
    };

    float2 S[CPL];  // S[j] = (S[r][c_j], S[r + 1][c_j]), c_j = cg * CPL + j
    if (active && a.init_state) {
        const float* s0 = a.init_state + (bh * dk + r) * (long)DV + cg * CPL;
        float x0[CPL], x1[CPL];
        load_run<CPL>(s0, x0);
        load_run<CPL>(s0 + DV, x1);
#pragma unroll
        for (int j = 0; j < CPL; j++) S[j] = make_float2(x0[j], x1[j]);
    } else {
#pragma unroll
        for (int j = 0; j < CPL; j++) S[j] = make_float2(0.f, 0.f);
    }

    // forward sweep: S_t and dq_t = S_t dout_t
    {
        const int n0 = min(kTB, L);
        fetch(0, n0, false);
        stage(n0, false, sm);
        __syncthreads();
        for (int t0 = 0, rnd = 0; t0 < L; t0 += kTB, rnd++) {
            const int n = min(kTB, L - t0);
            const int nn = min(kTB, L - t0 - kTB);
            if (nn > 0) fetch(t0 + kTB, nn, false);
            const float* buf = sm + (rnd & 1) * BUF;
            const float* s_v = buf;
            const float* s_d = s_v + kTB * St::ROW;
            const float* s_k = s_d + kTB * St::ROW;
            const float* s_a = s_k + kTB * kBlock;
            if (active) {
                for (int t = 0; t < n; t++) {
                    float vr[CPL], dr[CPL];
                    load_run<CPL>(s_v + t * St::ROW + cg * St::STRIDE, vr);
                    load_run<CPL>(s_d + t * St::ROW + cg * St::STRIDE, dr);
                    const float2 k2 = *reinterpret_cast<const float2*>(s_k + t * kBlock + rl);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
                    if (GATE) {
                        const float2 a2 = *reinterpret_cast<const float2*>(s_a + t * kBlock + rl);
#pragma unroll
                        for (int j = 0; j < CPL; j++) S[j] = fma2(a2, S[j], mul2(k2, dup(vr[j])));
                    } else {
#pragma unroll
                        for (int j = 0; j < CPL; j++) S[j] = fma2(k2, dup(vr[j]), S[j]);
                    }
#pragma unroll
                    for (int j = 0; j < CPL; j += 2) {
                        acc0 = fma2(S[j], dup(dr[j]), acc0);
                        acc1 = fma2(S[j + 1], dup(dr[j + 1]), acc1);
                    }
                    const float2 d = group_sum(make_float2(acc0.x + acc1.x, acc0.y + acc1.y));
                    if (cg == 0) *reinterpret_cast<float2*>(dq + (long)(t0 + t) * dk + r) = d;
                }
            }
            if (nn > 0) stage(nn, false, sm + ((rnd + 1) & 1) * BUF);
            __syncthreads();
        }
    }

    // the boundary term of the gate gradient: rowsum(dfinal * S_{L-1})
    float2 gsum = make_float2(0.f, 0.f);
    if (active) {
        const float* df = a.dfinal ? a.dfinal + (bh * dk + r) * (long)DV + cg * CPL : nullptr;
        float x0[CPL], x1[CPL];
        if (df) {
            load_run<CPL>(df, x0);
            load_run<CPL>(df + DV, x1);
        } else {
#pragma unroll
            for (int j = 0; j < CPL; j++) x0[j] = 0.f, x1[j] = 0.f;
        }
        if (GATE && df) {
            float2 c = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < CPL; j++) c = fma2(S[j], make_float2(x0[j], x1[j]), c);
            gsum = group_sum(c);
        }
        // from here S holds G, the gradient reaching the state (dfinal at t = L - 1)
#pragma unroll
        for (int j = 0; j < CPL; j++) S[j] = make_float2(x0[j], x1[j]);
    }

    // reverse sweep: G_t, dk_t = G_t v_t, dlog_alpha_t, then G <- Diag(alpha_t) G
    float* dkp = a.dk_out + bh * (long)L * dk;
    float* dla = GATE && a.dlog_alpha ? a.dlog_alpha + bh * (long)L * dk : nullptr;
    {
        const int nr = (L + kTB - 1) / kTB;  // rounds, the last one first
        auto span = [&](int rr, int& t0) {
            const int hi = L - rr * kTB;
            t0 = max(0, hi - kTB);
            return hi - t0;
        };
        int t0;
        int n = span(0, t0);
        fetch(t0, n, true);
        stage(n, true, sm);
        __syncthreads();
        for (int rr = 0; rr < nr; rr++) {
            n = span(rr, t0);
            int tn = 0, nn = 0;
            if (rr + 1 < nr) {
                nn = span(rr + 1, tn);
                fetch(tn, nn, true);
            }
            const float* buf = sm + (rr & 1) * BUF;
            const float* s_v = buf;
            const float* s_d = s_v + kTB * St::ROW;
            const float* s_k = s_d + kTB * St::ROW;
            const float* s_a = s_k + kTB * kBlock;
            const float* s_q = s_a + kTB * kBlock;
            const float* s_dq = s_q + kTB * kBlock;
            if (active) {
                for (int t = n - 1; t >= 0; t--) {
                    float vr[CPL], dr[CPL];
                    load_run<CPL>(s_v + t * St::ROW + cg * St::STRIDE, vr);
                    load_run<CPL>(s_d + t * St::ROW + cg * St::STRIDE, dr);
                    const float2 q2 = *reinterpret_cast<const float2*>(s_q + t * kBlock + rl);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
                    for (int j = 0; j < CPL; j += 2) {
                        S[j] = fma2(q2, dup(dr[j]), S[j]);
                        S[j + 1] = fma2(q2, dup(dr[j + 1]), S[j + 1]);
                        acc0 = fma2(S[j], dup(vr[j]), acc0);
                        acc1 = fma2(S[j + 1], dup(vr[j + 1]), acc1);
                    }
                    const float2 d = group_sum(make_float2(acc0.x + acc1.x, acc0.y + acc1.y));
                    const long o = (long)(t0 + t) * dk + r;
                    if (cg == 0) *reinterpret_cast<float2*>(dkp + o) = d;
                    if (GATE) {
                        const float2 a2 = *reinterpret_cast<const float2*>(s_a + t * kBlock + rl);
#pragma unroll
                        for (int j = 0; j < CPL; j++) S[j] = mul2(a2, S[j]);
                        const float2 k2 = *reinterpret_cast<const float2*>(s_k + t * kBlock + rl);
                        const float2 dq2 = *reinterpret_cast<const float2*>(s_dq + t * kBlock + rl);
                        // running sum over s >= t of q_s dq_s - k_s dk_s
                        gsum = fma2(q2, dq2, gsum);
                        gsum = fma2(make_float2(-k2.x, -k2.y), d, gsum);
                        if (dla && cg == 0) *reinterpret_cast<float2*>(dla + o) = gsum;
                    }
                }
            }
            if (nn > 0) stage(nn, true, sm + ((rr + 1) & 1) * BUF);
            __syncthreads();
        }
    }
    if (active && a.dinit) {
        float* di = a.dinit + (bh * dk + r) * (long)DV + cg * CPL;
#pragma unroll
        for (int j = 0; j < CPL; j++) {
            di[j] = S[j].x;
            di[DV + j] = S[j].y;
        }
    }
}

// ---- column CTAs: dv (reverse sweep) ----
// Wide arrays are over the key rows (W = RPL): q, k, alpha.  Narrow arrays over
// the CTA's 64 value columns: dout.
template <int RPL, bool GATE, typename T>
__device__ __forceinline__ void cols_body(const BwdArgs& a, float* sm, int blk) {
    using St = Stage<RPL>;
    constexpr int DK = St::FULL;
    constexpr int BUF = kTB * (3 * St::ROW + kBlock);
    const int L = a.L, dv = a.dv;
    const long bh = blockIdx.x;
    const int col0 = blk * kBlock, ncols = min(kBlock, dv - col0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 1, cp = lane & 1;
    const int c = warp * 4 + cp * 2;
    const bool active = warp * 4 < ncols;  // dv is a multiple of 4
    const int r0 = rg * RPL;

    const T* q = static_cast<const T*>(a.q) + bh * (long)L * DK;
    const T* k = static_cast<const T*>(a.k) + bh * (long)L * DK;
    const T* dout = static_cast<const T*>(a.dout) + bh * (long)L * dv;
    const float* la = GATE ? a.log_alpha + bh * (long)L * DK : nullptr;

    T rq[St::NW], rk[St::NW], rd[St::NN];
    float ra[St::NW];
    auto fetch = [&](int t0, int n) {
#pragma unroll
        for (int m = 0; m < St::NW; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DK) {
                const long g = (long)t0 * DK + idx;
                rq[m] = q[g];
                rk[m] = k[g];
                if (GATE) ra[m] = la[g];
            }
        }
#pragma unroll
        for (int m = 0; m < St::NN; m++) {
            const int idx = tid + m * kThreads;
            const int t = idx / kBlock, j = idx % kBlock;
            if (t < n && j < ncols) rd[m] = dout[(long)(t0 + t) * dv + col0 + j];
        }
    };
    auto stage = [&](int n, float* buf) {
        float* s_q = buf;
        float* s_k = s_q + kTB * St::ROW;
        float* s_a = s_k + kTB * St::ROW;
        float* s_d = s_a + kTB * St::ROW;
#pragma unroll
        for (int m = 0; m < St::NW; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DK) {
                const int o = (idx / DK) * St::ROW + St::pidx(idx % DK);
                s_q[o] = to_f(rq[m]);
                s_k[o] = to_f(rk[m]);
                s_a[o] = GATE ? __expf(ra[m]) : 1.f;
            }
        }
#pragma unroll
        for (int m = 0; m < St::NN; m++) {
            const int idx = tid + m * kThreads;
            if (idx / kBlock < n && idx % kBlock < ncols) s_d[idx] = to_f(rd[m]);
        }
    };

    float2 G[RPL];  // G[i] = (G[r0 + i][col0 + c], G[r0 + i][col0 + c + 1])
    if (active && a.dfinal) {
        const float* df = a.dfinal + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int i = 0; i < RPL; i++) G[i] = *reinterpret_cast<const float2*>(df + (long)(r0 + i) * dv);
    } else {
#pragma unroll
        for (int i = 0; i < RPL; i++) G[i] = make_float2(0.f, 0.f);
    }

    float* dvp = a.dv_out + bh * (long)L * dv + col0 + c;
    const int nr = (L + kTB - 1) / kTB;
    auto span = [&](int rr, int& t0) {
        const int hi = L - rr * kTB;
        t0 = max(0, hi - kTB);
        return hi - t0;
    };
    int t0;
    int n = span(0, t0);
    fetch(t0, n);
    stage(n, sm);
    __syncthreads();
    for (int rr = 0; rr < nr; rr++) {
        n = span(rr, t0);
        int tn = 0, nn = 0;
        if (rr + 1 < nr) {
            nn = span(rr + 1, tn);
            fetch(tn, nn);
        }
        const float* buf = sm + (rr & 1) * BUF;
        const float* s_q = buf;
        const float* s_k = s_q + kTB * St::ROW;
        const float* s_a = s_k + kTB * St::ROW;
        const float* s_d = s_a + kTB * St::ROW;
        if (active) {
            for (int t = n - 1; t >= 0; t--) {
                const int ro = t * St::ROW + rg * St::STRIDE;
                float qr[RPL], kr[RPL];
                load_run<RPL>(s_q + ro, qr);
                load_run<RPL>(s_k + ro, kr);
                const float2 d2 = *reinterpret_cast<const float2*>(s_d + t * kBlock + c);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
                for (int i = 0; i < RPL; i += 2) {
                    G[i] = fma2(dup(qr[i]), d2, G[i]);
                    G[i + 1] = fma2(dup(qr[i + 1]), d2, G[i + 1]);
                    acc0 = fma2(dup(kr[i]), G[i], acc0);
                    acc1 = fma2(dup(kr[i + 1]), G[i + 1], acc1);
                }
                const float2 d = group_sum(make_float2(acc0.x + acc1.x, acc0.y + acc1.y));
                if (rg == 0) *reinterpret_cast<float2*>(dvp + (long)(t0 + t) * dv) = d;
                if (GATE) {
                    float ar[RPL];
                    load_run<RPL>(s_a + ro, ar);
#pragma unroll
                    for (int i = 0; i < RPL; i++) G[i] = mul2(G[i], dup(ar[i]));
                }
            }
        }
        if (nn > 0) stage(nn, sm + ((rr + 1) & 1) * BUF);
        __syncthreads();
    }
}

template <int CPL, int RPL>
constexpr size_t bwd_smem_bytes() {
    constexpr size_t rows = (size_t)kTB * (2 * Stage<CPL>::ROW + 4 * kBlock);
    constexpr size_t cols = (size_t)kTB * (3 * Stage<RPL>::ROW + kBlock);
    return sizeof(float) * 2 * (rows > cols ? rows : cols);
}

// blockIdx.x: (batch, head); blockIdx.y < row_blocks: a row CTA, else a column CTA
template <int CPL, int RPL, bool GATE, typename T>
__global__ void __launch_bounds__(kThreads) gla_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int row_blocks = (a.dk + kBlock - 1) / kBlock;
    if ((int)blockIdx.y < row_blocks)
        rows_body<CPL, GATE, T>(a, sm, blockIdx.y);
    else
        cols_body<RPL, GATE, T>(a, sm, blockIdx.y - row_blocks);
}

template <int CPL, int RPL, bool GATE, typename T>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t s) {
    auto kern = gla_bwd_kernel<CPL, RPL, GATE, T>;
    constexpr size_t smem = bwd_smem_bytes<CPL, RPL>();
    static_assert(smem <= 227 * 1024, "staging exceeds shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned rb = (unsigned)((a.dk + kBlock - 1) / kBlock), cb = (unsigned)((a.dv + kBlock - 1) / kBlock);
    const dim3 grid((unsigned)((long)a.B * a.H), rb + cb);
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int CPL, int RPL>
cudaError_t launch_g(const BwdArgs& a, cudaStream_t s) {
    const bool bf = a.in_dtype == GLA_DTYPE_BF16;
    if (a.log_alpha)
        return bf ? launch_t<CPL, RPL, true, __nv_bfloat16>(a, s) : launch_t<CPL, RPL, true, float>(a, s);
    return bf ? launch_t<CPL, RPL, false, __nv_bfloat16>(a, s) : launch_t<CPL, RPL, false, float>(a, s);
}

template <int CPL>
cudaError_t launch_dk(const BwdArgs& a, cudaStream_t s) {
    switch (a.dk) {
        case 32: return launch_g<CPL, 2>(a, s);
        case 64: return launch_g<CPL, 4>(a, s);
        default: return launch_g<CPL, 8>(a, s);
    }
}

}  // namespace

bool bwd_supported(int dk, int dv) {
    return (dk == 32 || dk == 64 || dk == 128) && (dv == 32 || dv == 64 || dv == 128);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s) {
    if ((long)a.B * a.H == 0 || a.L == 0) return cudaSuccess;
    switch (a.dv) {
        case 32: return launch_dk<2>(a, s);
        case 64: return launch_dk<4>(a, s);
        default: return launch_dk<8>(a, s);
    }
}

}  // namespace gla
