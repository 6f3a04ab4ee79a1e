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
// are the only place log alpha appears.)  With one gate per token
// (GLA_FLAG_SCALAR_GATE) every row stages the token's alpha, and the token's
// gradient is the sum of the rows' (warp shuffles, then fp32 atomics across
// the row CTAs of a head).
//
// Two kinds of CTA share one launch:
//  * row CTAs own 32 key rows of one head, all value columns.  Rows evolve on
//    their own (S_t[i,:] needs alpha_t[i], k_t[i] and v_t), so a forward sweep
//    carries S and emits dq (a reduction over the value columns), and a
//    reverse sweep carries G and emits dk, the running gate sum and dS_{-1}.
//    Lane (cg, rp) of a warp holds rows warp*4 + 2 rp + {0, 1} over the value
//    columns [cg * CPL, (cg + 1) * CPL), as fp32 pairs of adjacent columns.
//  * column CTAs own 32 value columns: a reverse sweep carries G column-wise
//    and emits dv (a reduction over the key rows).  Lane (rg, cp) holds rows
//    [rg * RPL, (rg + 1) * RPL) of the columns 2 cp + {0, 1}, as fp32 pairs of
//    adjacent rows.
// Pairs run along the vectors read from shared memory per token, so they feed
// the packed fp32 instructions as loaded; the per-lane scalars (k, alpha, q of
// a row, dout of a column) are staged as (x, x) pairs.  The reductions are
// output-only (they do not feed the recurrence), so a batch of 8 tokens keeps
// its 16 partial sums per lane and reduce-scatters them across the sixteen
// lane groups.  Rounds of 16 tokens are staged in shared memory, double
// buffered: the next round's global loads are in flight while the current one
// is computed.  8 warps and at most 128 registers per thread give two CTAs per
// SM; row CTAs come first in the grid (they do two sweeps, the column CTAs
// one), the row blocks of a head adjacent so that they share its v and dout
// through L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTB = 16;             // tokens staged per round
constexpr int kRB = 8;              // tokens per batch of reductions
constexpr int kBlock = 4 * kWarps;  // rows per row CTA, columns per column CTA

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

// sum over the sixteen lane groups (lane bits 1..4), every lane gets the total
__device__ __forceinline__ float2 group_sum(float2 x) {
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, m);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, m);
    }
    return x;
}

// Reduce-scatter over the sixteen lane groups: v[e] (e = 2 tb + w, 16 partial
// sums per lane) summed across lane bits 1..4; lane group g = lane >> 1 ends
// with the total of entry e = g.  Four halving exchanges: 15 shuffles for 16
// sums instead of 64.
__device__ __forceinline__ float reduce_scatter16(const float2 (&acc)[kRB], int lane) {
    float v8[8];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float lo = i & 1 ? acc[i >> 1].y : acc[i >> 1].x;
            const float hi = i & 1 ? acc[4 + (i >> 1)].y : acc[4 + (i >> 1)].x;
            const float send = up ? lo : hi, mine = up ? hi : lo;
            v8[i] = mine + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    float v4[4];
    {
        const bool up = lane & 8;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float send = up ? v8[i] : v8[4 + i], mine = up ? v8[4 + i] : v8[i];
            v4[i] = mine + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    float v2[2];
    {
        const bool up = lane & 4;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const float send = up ? v4[i] : v4[2 + i], mine = up ? v4[2 + i] : v4[i];
            v2[i] = mine + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    }
    const bool up = lane & 2;
    const float send = up ? v2[0] : v2[1], mine = up ? v2[1] : v2[0];
    return mine + __shfl_xor_sync(0xffffffffu, send, 2);
}

template <typename T>
__device__ __forceinline__ float to_f(T x) {
    if constexpr (std::is_same<T, float>::value)
        return x;
    else
        return __bfloat162float(x);
}

// N consecutive floats of a staged group as N / 2 pairs (16-byte aligned when N >= 4)
template <int N>
__device__ __forceinline__ void load_pairs(const float* p, float2 (&r)[N / 2]) {
    if constexpr (N >= 4) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + i);
            r[i / 2] = make_float2(x.x, x.y);
            r[i / 2 + 1] = make_float2(x.z, x.w);
        }
    } else {
        r[0] = *reinterpret_cast<const float2*>(p);
    }
}

// Staging of one round of tokens.  "Wide" arrays span the full dimension that
// the CTA's lanes split in sixteen groups of W floats (padded to W + 4 per
// group); "narrow" arrays span only the CTA's own kBlock entries.
template <int W>
struct Stage {
    static constexpr int FULL = 16 * W;
    static constexpr int STRIDE = W + 4;
    static constexpr int ROW = 16 * STRIDE;
    __device__ static constexpr int pidx(int x) { return (x / W) * STRIDE + x % W; }
    static constexpr int NW = (kTB * FULL + kThreads - 1) / kThreads;    // wide loads per thread
    static constexpr int NN = (kTB * kBlock + kThreads - 1) / kThreads;  // narrow loads per thread
};

// rounds of the reverse sweeps: the last kTB tokens first; returns the count, sets t0
__device__ __forceinline__ int rev_span(int L, int rr, int& t0) {
    const int hi = L - rr * kTB;
    t0 = max(0, hi - kTB);
    return hi - t0;
}

// ---- row CTAs: dq (forward sweep); dk, dlog_alpha, dS_{-1} (reverse sweep) ----
// Wide arrays are over the value columns (W = CPL): v, dout.  Narrow arrays over
// the CTA's key rows: k, alpha, and q, dq in the reverse sweep.  A lane's state
// is S[w][p] = (S[r + w][c_{2p}], S[r + w][c_{2p+1}]), w = 0, 1, c_j = cg CPL + j.
template <int CPL, bool GATE, typename T>
__device__ __forceinline__ void rows_body(const BwdArgs& a, float* sm, long bh, int blk) {
    using St = Stage<CPL>;
    constexpr int DV = St::FULL, NP = CPL / 2;
    constexpr int BUF = kTB * (2 * St::ROW + 7 * kBlock);
    const int L = a.L, dk = a.dk;
    const int row0 = blk * kBlock, nrows = min(kBlock, dk - row0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = lane >> 1, rp = lane & 1;
    const int rl = warp * 4 + rp * 2;      // this lane's first row within the block
    const bool active = warp * 4 < nrows;  // dk is a multiple of 4: a warp is all or nothing
    const int r = row0 + rl;
    // after a reduce-scatter this lane holds token tb_l of row rl + w_l
    const int tb_l = cg >> 1, w_l = cg & 1;

    const T* q = static_cast<const T*>(a.q) + bh * (long)L * dk;
    const T* k = static_cast<const T*>(a.k) + bh * (long)L * dk;
    const T* v = static_cast<const T*>(a.v) + bh * (long)L * DV;
    const T* dout = static_cast<const T*>(a.dout) + bh * (long)L * DV;
    // per-channel gate [L][dk]; per-token gate (GLA_FLAG_SCALAR_GATE) [L], shared by all rows
    const bool scalar = a.flags & GLA_FLAG_SCALAR_GATE;
    const float* la = GATE ? a.log_alpha + bh * (long)L * (scalar ? 1 : dk) : nullptr;
    float* dq = a.dq + bh * (long)L * dk;

    T rv[St::NW], rd[St::NW], rk[St::NN], rq[St::NN];
    float ra[St::NN], rdq[St::NN];
    // round [t0, t0 + n): global -> registers; rev also fetches q and dq
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
                if (GATE) ra[m] = scalar ? la[t0 + t] : la[g];
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
        float2* s_k = reinterpret_cast<float2*>(s_d + kTB * St::ROW);  // (k, k) per entry
        float2* s_a = s_k + kTB * kBlock;                               // (alpha, alpha)
        float2* s_q = s_a + kTB * kBlock;                               // (q, q)
        float* s_dq = reinterpret_cast<float*>(s_q + kTB * kBlock);
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
                s_k[idx] = dup(to_f(rk[m]));
                s_a[idx] = dup(GATE ? __expf(ra[m]) : 1.f);
                if (rev) {
                    s_q[idx] = dup(to_f(rq[m]));
                    s_dq[idx] = GATE ? rdq[m] : 0.f;
                }
            }
        }
    };

    float2 S[2][NP];
    if (active && a.init_state) {
        const float* s0 = a.init_state + (bh * dk + r) * (long)DV + cg * CPL;
        load_pairs<CPL>(s0, S[0]);
        load_pairs<CPL>(s0 + DV, S[1]);
    } else {
#pragma unroll
        for (int w = 0; w < 2; w++)
#pragma unroll
            for (int p = 0; p < NP; p++) S[w][p] = make_float2(0.f, 0.f);
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
            const float* s_a = s_k + 2 * kTB * kBlock;
            if (active) {
#pragma unroll
                for (int h = 0; h < kTB / kRB; h++) {
                    float2 acc[kRB];
#pragma unroll
                    for (int u = 0; u < kRB; u++) {
                        const int t = h * kRB + u;
                        acc[u] = make_float2(0.f, 0.f);
                        if (t < n) {
                            float2 vp[NP], dp[NP];
                            load_pairs<CPL>(s_v + t * St::ROW + cg * St::STRIDE, vp);
                            load_pairs<CPL>(s_d + t * St::ROW + cg * St::STRIDE, dp);
                            const float4 k4 = *reinterpret_cast<const float4*>(s_k + 2 * (t * kBlock + rl));
                            const float4 a4 = *reinterpret_cast<const float4*>(s_a + 2 * (t * kBlock + rl));
                            float2 pr[2];
#pragma unroll
                            for (int w = 0; w < 2; w++) {
                                const float2 kd = w ? make_float2(k4.z, k4.w) : make_float2(k4.x, k4.y);
                                const float2 ad = w ? make_float2(a4.z, a4.w) : make_float2(a4.x, a4.y);
                                pr[w] = make_float2(0.f, 0.f);
#pragma unroll
                                for (int p = 0; p < NP; p++) {
                                    S[w][p] = GATE ? fma2(ad, S[w][p], mul2(kd, vp[p])) : fma2(kd, vp[p], S[w][p]);
                                    pr[w] = fma2(S[w][p], dp[p], pr[w]);
                                }
                            }
                            acc[u] = make_float2(pr[0].x + pr[0].y, pr[1].x + pr[1].y);
                        }
                    }
                    const float x = reduce_scatter16(acc, lane);
                    const int tt = h * kRB + tb_l;
                    if (tt < n) dq[(long)(t0 + tt) * dk + r + w_l] = x;
                }
            }
            if (nn > 0) stage(nn, false, sm + ((rnd + 1) & 1) * BUF);
            __syncthreads();
        }
    }

    // the boundary term of the gate gradient, rowsum(dfinal * S_{L-1}), for row rl + w_l
    float carry = 0.f;
    if (active) {
        const float* df = a.dfinal ? a.dfinal + (bh * dk + r) * (long)DV + cg * CPL : nullptr;
        float2 F[2][NP];
        if (df) {
            load_pairs<CPL>(df, F[0]);
            load_pairs<CPL>(df + DV, F[1]);
        } else {
#pragma unroll
            for (int w = 0; w < 2; w++)
#pragma unroll
                for (int p = 0; p < NP; p++) F[w][p] = make_float2(0.f, 0.f);
        }
        if (GATE && df) {
            float2 c[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int w = 0; w < 2; w++)
#pragma unroll
                for (int p = 0; p < NP; p++) c[w] = fma2(S[w][p], F[w][p], c[w]);
            const float2 cs = group_sum(make_float2(c[0].x + c[0].y, c[1].x + c[1].y));
            carry = w_l ? cs.y : cs.x;
        }
        // from here S holds G, the gradient reaching the state (dfinal at t = L - 1)
#pragma unroll
        for (int w = 0; w < 2; w++)
#pragma unroll
            for (int p = 0; p < NP; p++) S[w][p] = F[w][p];
    }

    // reverse sweep: G_t = G + q_t dout_t^T, dk_t = G_t v_t, the gate gradient, G <- Diag(alpha_t) G_t
    float* dkp = a.dk_out + bh * (long)L * dk;
    float* dla = GATE && a.dlog_alpha ? a.dlog_alpha + bh * (long)L * (scalar ? 1 : dk) : nullptr;
    {
        const int nr = (L + kTB - 1) / kTB;
        int t0;
        int n = rev_span(L, 0, t0);
        fetch(t0, n, true);
        stage(n, true, sm);
        __syncthreads();
        for (int rr = 0; rr < nr; rr++) {
            n = rev_span(L, rr, t0);
            int tn = 0, nn = 0;
            if (rr + 1 < nr) {
                nn = rev_span(L, rr + 1, tn);
                fetch(tn, nn, true);
            }
            const float* buf = sm + (rr & 1) * BUF;
            const float* s_v = buf;
            const float* s_d = s_v + kTB * St::ROW;
            const float* s_k = s_d + kTB * St::ROW;
            const float* s_a = s_k + 2 * kTB * kBlock;
            const float* s_q = s_a + 2 * kTB * kBlock;
            const float* s_dq = s_q + 2 * kTB * kBlock;
            if (active) {
#pragma unroll
                for (int h = kTB / kRB - 1; h >= 0; h--) {
                    float2 acc[kRB];
#pragma unroll
                    for (int u = kRB - 1; u >= 0; u--) {
                        const int t = h * kRB + u;
                        acc[u] = make_float2(0.f, 0.f);
                        if (t < n) {
                            float2 vp[NP], dp[NP];
                            load_pairs<CPL>(s_v + t * St::ROW + cg * St::STRIDE, vp);
                            load_pairs<CPL>(s_d + t * St::ROW + cg * St::STRIDE, dp);
                            const float4 q4 = *reinterpret_cast<const float4*>(s_q + 2 * (t * kBlock + rl));
                            const float4 a4 = *reinterpret_cast<const float4*>(s_a + 2 * (t * kBlock + rl));
                            float2 pr[2];
#pragma unroll
                            for (int w = 0; w < 2; w++) {
                                const float2 qd = w ? make_float2(q4.z, q4.w) : make_float2(q4.x, q4.y);
                                const float2 ad = w ? make_float2(a4.z, a4.w) : make_float2(a4.x, a4.y);
                                pr[w] = make_float2(0.f, 0.f);
#pragma unroll
                                for (int p = 0; p < NP; p++) {
                                    S[w][p] = fma2(qd, dp[p], S[w][p]);
                                    pr[w] = fma2(S[w][p], vp[p], pr[w]);
                                    if (GATE) S[w][p] = mul2(ad, S[w][p]);
                                }
                            }
                            acc[u] = make_float2(pr[0].x + pr[0].y, pr[1].x + pr[1].y);
                        }
                    }
                    const float x = reduce_scatter16(acc, lane);  // dk of token h kRB + tb_l, row rl + w_l
                    const int tt = h * kRB + tb_l;
                    const bool ok = tt < n;
                    const long o = (long)(t0 + tt) * dk + r + w_l;
                    if (ok) dkp[o] = x;
                    if (GATE) {
                        // suffix sums over the batch's tokens of q dq - k dk, plus the later tokens' total
                        const int i = tt * kBlock + rl + w_l;
                        float s = ok ? fmaf(s_q[2 * i], s_dq[i], -s_k[2 * i] * x) : 0.f;
#pragma unroll
                        for (int d = 1; d < kRB; d <<= 1) {
                            const float o2 = __shfl_down_sync(0xffffffffu, s, 4 * d);
                            if (tb_l + d < kRB) s += o2;
                        }
                        const float total = __shfl_sync(0xffffffffu, s, lane & 3);  // the batch's first token
                        if (!scalar) {
                            if (dla && ok) dla[o] = s + carry;
                        } else if (dla) {
                            // a per-token gate's gradient is the sum over all rows: this warp's four
                            // rows here (lanes 4 tb + {0..3}), the row blocks through atomics
                            float g4 = s + carry;
                            g4 += __shfl_xor_sync(0xffffffffu, g4, 1);
                            g4 += __shfl_xor_sync(0xffffffffu, g4, 2);
                            if (ok && (lane & 3) == 0) atomicAdd(dla + t0 + tt, g4);
                        }
                        carry += total;
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
        for (int w = 0; w < 2; w++)
#pragma unroll
            for (int p = 0; p < NP; p++) *reinterpret_cast<float2*>(di + w * DV + 2 * p) = S[w][p];
    }
}

// ---- column CTAs: dv (reverse sweep) ----
// Wide arrays are over the key rows (W = RPL): q, k, alpha.  Narrow arrays over
// the CTA's value columns: dout.  A lane's state is G[w][p] = (G[r0 + 2p][c + w],
// G[r0 + 2p + 1][c + w]), w = 0, 1.
template <int RPL, bool GATE, typename T>
__device__ __forceinline__ void cols_body(const BwdArgs& a, float* sm, long bh, int blk) {
    using St = Stage<RPL>;
    constexpr int DK = St::FULL, NP = RPL / 2;
    constexpr int BUF = kTB * (3 * St::ROW + 2 * kBlock);
    const int L = a.L, dv = a.dv;
    const int col0 = blk * kBlock, ncols = min(kBlock, dv - col0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 1, cp = lane & 1;
    const int c = warp * 4 + cp * 2;
    const bool active = warp * 4 < ncols;  // dv is a multiple of 4
    const int r0 = rg * RPL;
    const int tb_l = rg >> 1, w_l = rg & 1;

    const T* q = static_cast<const T*>(a.q) + bh * (long)L * DK;
    const T* k = static_cast<const T*>(a.k) + bh * (long)L * DK;
    const T* dout = static_cast<const T*>(a.dout) + bh * (long)L * dv;
    const bool scalar = a.flags & GLA_FLAG_SCALAR_GATE;
    const float* la = GATE ? a.log_alpha + bh * (long)L * (scalar ? 1 : DK) : nullptr;

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
                if (GATE) ra[m] = scalar ? la[t0 + idx / DK] : la[g];
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
        float2* s_d = reinterpret_cast<float2*>(s_a + kTB * St::ROW);  // (dout, dout) per entry
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
            if (idx / kBlock < n && idx % kBlock < ncols) s_d[idx] = dup(to_f(rd[m]));
        }
    };

    float2 G[2][NP];
    if (active && a.dfinal) {
        const float* df = a.dfinal + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int p = 0; p < NP; p++) {
            const float2 x0 = *reinterpret_cast<const float2*>(df + (long)(r0 + 2 * p) * dv);
            const float2 x1 = *reinterpret_cast<const float2*>(df + (long)(r0 + 2 * p + 1) * dv);
            G[0][p] = make_float2(x0.x, x1.x);
            G[1][p] = make_float2(x0.y, x1.y);
        }
    } else {
#pragma unroll
        for (int w = 0; w < 2; w++)
#pragma unroll
            for (int p = 0; p < NP; p++) G[w][p] = make_float2(0.f, 0.f);
    }

    float* dvp = a.dv_out + bh * (long)L * dv + col0 + c + w_l;
    const int nr = (L + kTB - 1) / kTB;
    int t0;
    int n = rev_span(L, 0, t0);
    fetch(t0, n);
    stage(n, sm);
    __syncthreads();
    for (int rr = 0; rr < nr; rr++) {
        n = rev_span(L, rr, t0);
        int tn = 0, nn = 0;
        if (rr + 1 < nr) {
            nn = rev_span(L, rr + 1, tn);
            fetch(tn, nn);
        }
        const float* buf = sm + (rr & 1) * BUF;
        const float* s_q = buf;
        const float* s_k = s_q + kTB * St::ROW;
        const float* s_a = s_k + kTB * St::ROW;
        const float* s_d = s_a + kTB * St::ROW;  // (dout, dout) pairs
        if (active) {
#pragma unroll
            for (int h = kTB / kRB - 1; h >= 0; h--) {
                float2 acc[kRB];
#pragma unroll
                for (int u = kRB - 1; u >= 0; u--) {
                    const int t = h * kRB + u;
                    acc[u] = make_float2(0.f, 0.f);
                    if (t < n) {
                        const int ro = t * St::ROW + rg * St::STRIDE;
                        float2 qp[NP], kp[NP];
                        load_pairs<RPL>(s_q + ro, qp);
                        load_pairs<RPL>(s_k + ro, kp);
                        const float4 d4 = *reinterpret_cast<const float4*>(s_d + 2 * (t * kBlock + c));
                        float2 ap[NP];
                        if (GATE) load_pairs<RPL>(s_a + ro, ap);
                        float2 pr[2];
#pragma unroll
                        for (int w = 0; w < 2; w++) {
                            const float2 dd = w ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
                            pr[w] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int p = 0; p < NP; p++) {
                                G[w][p] = fma2(qp[p], dd, G[w][p]);
                                pr[w] = fma2(kp[p], G[w][p], pr[w]);
                                if (GATE) G[w][p] = mul2(G[w][p], ap[p]);
                            }
                        }
                        acc[u] = make_float2(pr[0].x + pr[0].y, pr[1].x + pr[1].y);
                    }
                }
                const float x = reduce_scatter16(acc, lane);  // dv of token h kRB + tb_l, column c + w_l
                const int tt = h * kRB + tb_l;
                if (tt < n) dvp[(long)(t0 + tt) * dv] = x;
            }
        }
        if (nn > 0) stage(nn, sm + ((rr + 1) & 1) * BUF);
        __syncthreads();
    }
}

template <int CPL, int RPL>
constexpr size_t bwd_smem_bytes() {
    constexpr size_t rows = (size_t)kTB * (2 * Stage<CPL>::ROW + 7 * kBlock);
    constexpr size_t cols = (size_t)kTB * (3 * Stage<RPL>::ROW + 2 * kBlock);
    return sizeof(float) * 2 * (rows > cols ? rows : cols);
}

// 1-D grid: the first B H rb CTAs are row CTAs (the rb row blocks of a head
// adjacent, so they share its v and dout through L2), then B H cb column CTAs.
template <int CPL, int RPL, bool GATE, typename T>
__global__ void __launch_bounds__(kThreads, 2) gla_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const long BH = (long)a.B * a.H;
    const int rb = (a.dk + kBlock - 1) / kBlock, cb = (a.dv + kBlock - 1) / kBlock;
    const long b = blockIdx.x;
    if (a.only_marked) {
        // after the chunk-form backward: only the blocks of the heads it marked
        const uint32_t* mk = b < BH * rb
                                 ? reinterpret_cast<const uint32_t*>(a.dk_out) + (b / rb) * a.L * a.dk + (b % rb) * kBlock
                                 : reinterpret_cast<const uint32_t*>(a.dv_out) + ((b - BH * rb) / cb) * a.L * a.dv +
                                       ((b - BH * rb) % cb) * kBlock;
        if (*mk != kBwdMark) return;
    }
    if (b < BH * rb)
        rows_body<CPL, GATE, T>(a, sm, b / rb, (int)(b % rb));
    else
        cols_body<RPL, GATE, T>(a, sm, (b - BH * rb) / cb, (int)((b - BH * rb) % cb));
}

template <int CPL, int RPL, bool GATE, typename T>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t s) {
    auto kern = gla_bwd_kernel<CPL, RPL, GATE, T>;
    constexpr size_t smem = bwd_smem_bytes<CPL, RPL>();
    static_assert(smem <= 227 * 1024, "staging exceeds shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long blocks = (long)a.B * a.H * (bwd_blocks(a.dk) + bwd_blocks(a.dv));
    kern<<<(unsigned)blocks, kThreads, smem, s>>>(a);
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

int bwd_blocks(int d) { return (d + kBlock - 1) / kBlock; }

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
