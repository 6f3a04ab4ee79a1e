// gla_delta.cu -- the delta rule, token by token, on the GPU.
//
// "linear-attention" blog, Delta attention: before writing, the memory is
// asked what it already predicts for the key, and only the error is written,
// with a write strength beta_n:
//   p_n = S_{n-1}^T k_n,  u_n = beta_n (v_n - p_n),  S_n = S_{n-1} + k_n u_n^T,
//   o_n = S_n^T q_n;
// the gated variant first decays the state, S_{n-1} <- Diag(alpha_n) S_{n-1}.
//
// Each value column of the state evolves on its own (p_n, u_n and the write
// are column-wise given k_n and beta_n), so a warp owns 4 value columns of one
// head for the whole sequence and needs no block-wide synchronisation per
// token: lane (rg, cp) holds rows [rg * RPL, (rg + 1) * RPL) of the column
// pair 2 cp (RPL = dk / 16 rows, as packed fp32 pairs).  The prediction is a
// reduction over dk that feeds the write, so it takes four butterfly shuffles
// across the sixteen row groups every token; the output does not feed the
// recurrence, so a batch of 4 tokens keeps its partial sums and
// reduce-scatters them (8 shuffles for 4 tokens instead of 32).  A CTA of 16
// warps covers 64 value columns, two CTAs per SM (64 registers); tokens are
// staged in shared memory 16 at a time, double buffered: the next round's
// global loads are in flight while the current round is computed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kWarps = 16;            // 4 value columns each
constexpr int kCols = 4 * kWarps;     // value columns per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kTB = 16;               // tokens staged per round
constexpr int kRB = 4;                // tokens per batch of output reductions

template <int RPL>
struct DeltaLayout {
    static constexpr int DK = RPL * 16;
    static constexpr int STRIDE = RPL + 4;   // padded floats per row group (16-byte aligned for RPL >= 4)
    static constexpr int ROW = 16 * STRIDE;  // padded floats per token
    __host__ __device__ static constexpr int pidx(int r) { return (r / RPL) * STRIDE + r % RPL; }
    static constexpr int BUF = kTB * (3 * ROW + kCols + 4);  // floats per staging buffer
    static constexpr size_t bytes = sizeof(float) * 2 * (size_t)BUF;
    // elements of one round each thread loads: q, k, log alpha (DK per token) and v (kCols per token)
    static constexpr int NQ = (kTB * DK + kThreads - 1) / kThreads;
    static constexpr int NV = (kTB * kCols + kThreads - 1) / kThreads;
};

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

// sum over the sixteen row groups (lane bits 1..4)
__device__ __forceinline__ float2 rowgroup_sum(float2 x) {
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, m);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, m);
    }
    return x;
}

// Reduce-scatter over the sixteen row groups (lane bits 1..4) of the 2 NB partial
// sums of a lane (entry e = 2 tb + w): halving exchanges while entries remain,
// then plain butterfly adds.  NB = 8: row group g ends with entry g; NB = 4:
// row groups 2e and 2e + 1 both end with entry e.
template <int NB>
__device__ __forceinline__ float reduce_scatter(const float2 (&acc)[NB], int lane) {
    float v[2 * NB];
#pragma unroll
    for (int i = 0; i < NB; i++) v[2 * i] = acc[i].x, v[2 * i + 1] = acc[i].y;
    int n = 2 * NB;
#pragma unroll
    for (int mask = 16; mask >= 2; mask >>= 1) {
        if (n > 1) {
            const bool up = lane & mask;
            const int half = n / 2;
#pragma unroll
            for (int i = 0; i < half; i++) {
                const float send = up ? v[i] : v[half + i], mine = up ? v[half + i] : v[i];
                v[i] = mine + __shfl_xor_sync(0xffffffffu, send, mask);
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
    }
    return v[0];
}

// RPL consecutive floats of a staged row group (16-byte aligned when RPL >= 4)
template <int RPL>
__device__ __forceinline__ void load_rows(const float* p, float (&r)[RPL]) {
    if constexpr (RPL >= 4) {
#pragma unroll
        for (int i = 0; i < RPL; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + i);
            r[i] = x.x, r[i + 1] = x.y, r[i + 2] = x.z, r[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < RPL; i += 2) {
            const float2 x = *reinterpret_cast<const float2*>(p + i);
            r[i] = x.x, r[i + 1] = x.y;
        }
    }
}

template <int RPL, bool GATE, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 2) gla_delta_kernel(const DeltaArgs a) {
    using Ly = DeltaLayout<RPL>;
    constexpr int DK = Ly::DK;
    extern __shared__ __align__(16) float sm[];

    const int L = a.L, dv = a.dv;
    const long bh = blockIdx.x;
    const int col0 = blockIdx.y * kCols;
    const int ncols = min(kCols, dv - col0);
    if (a.only_marked) {
        // after the chunk-form kernel: only the column blocks of the heads it marked
        const long m = bh * L * dv + col0;
        const bool marked = a.out_dtype == GLA_DTYPE_F32
                                ? reinterpret_cast<const uint32_t*>(a.out)[m] == kDeltaMarkF32
                                : reinterpret_cast<const uint16_t*>(a.out)[m] == kDeltaMarkBf16;
        if (!marked) return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 1, cp = lane & 1;
    const int c = warp * 4 + cp * 2;        // this lane's first column within the CTA's block
    const bool active = c < ncols;          // dv is a multiple of 16: a warp is all or nothing
    const int r0 = rg * RPL;
    // after a reduce-scatter: token tb_l of the batch, column c + w_l (two row groups hold each)
    const int tb_l = rg >> 2, w_l = (rg >> 1) & 1;
    const bool writer = (rg & 1) == 0;

    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + bh * (long)L * DK;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + bh * (long)L * DK;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + bh * (long)L * dv;
    const float* la = GATE ? a.log_alpha + bh * (long)L * DK : nullptr;
    const float* beta = a.beta + bh * (long)L;

    // one round of tokens [t0, t0 + n): global -> registers, registers -> a staging buffer
    __nv_bfloat16 rq[Ly::NQ], rk[Ly::NQ];
    float ra[Ly::NQ];
    __nv_bfloat16 rv[Ly::NV];
    float rb = 0.f;
    auto fetch = [&](int t0) {
        const int n = min(kTB, L - t0);
#pragma unroll
        for (int m = 0; m < Ly::NQ; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DK) {
                const long g = (long)t0 * DK + idx;
                rq[m] = q[g];
                rk[m] = k[g];
                if (GATE) ra[m] = la[g];
            }
        }
#pragma unroll
        for (int m = 0; m < Ly::NV; m++) {
            const int idx = tid + m * kThreads;
            const int t = idx / kCols, j = idx % kCols;
            if (t < n && j < ncols) rv[m] = v[(long)(t0 + t) * dv + col0 + j];
        }
        if (tid < n) rb = beta[t0 + tid];
    };
    auto stage = [&](int t0, float* buf) {
        const int n = min(kTB, L - t0);
        float* s_q = buf;
        float* s_k = s_q + kTB * Ly::ROW;
        float* s_a = s_k + kTB * Ly::ROW;
        float* s_v = s_a + kTB * Ly::ROW;
        float* s_b = s_v + kTB * kCols;
#pragma unroll
        for (int m = 0; m < Ly::NQ; m++) {
            const int idx = tid + m * kThreads;
            if (idx < n * DK) {
                const int o = (idx / DK) * Ly::ROW + Ly::pidx(idx % DK);
                s_q[o] = __bfloat162float(rq[m]);
                s_k[o] = __bfloat162float(rk[m]);
                if (GATE) s_a[o] = __expf(ra[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < Ly::NV; m++) {
            const int idx = tid + m * kThreads;
            const int t = idx / kCols, j = idx % kCols;
            if (t < n && j < ncols) s_v[t * kCols + j] = __bfloat162float(rv[m]);
        }
        if (tid < n) s_b[tid] = rb;
    };

    float2 S[RPL];
    if (active && a.init_state) {
        const float* s0 = a.init_state + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int i = 0; i < RPL; i++) S[i] = *reinterpret_cast<const float2*>(s0 + (long)(r0 + i) * dv);
    } else {
#pragma unroll
        for (int i = 0; i < RPL; i++) S[i] = make_float2(0.f, 0.f);
    }

    fetch(0);
    stage(0, sm);
    __syncthreads();
    for (int t0 = 0, rnd = 0; t0 < L; t0 += kTB, rnd++) {
        const int n = min(kTB, L - t0);
        const bool more = t0 + kTB < L;
        if (more) fetch(t0 + kTB);  // in flight while this round is computed
        const float* buf = sm + (rnd & 1) * Ly::BUF;
        const float* s_q = buf;
        const float* s_k = s_q + kTB * Ly::ROW;
        const float* s_a = s_k + kTB * Ly::ROW;
        const float* s_v = s_a + kTB * Ly::ROW;
        const float* s_b = s_v + kTB * kCols;
        if (active) {
#pragma unroll
            for (int h = 0; h < kTB / kRB; h++) {
                float2 acc[kRB];
#pragma unroll
                for (int uu = 0; uu < kRB; uu++) {
                    const int t = h * kRB + uu;
                    acc[uu] = make_float2(0.f, 0.f);
                    if (t < n) {
                        const int ro = t * Ly::ROW + rg * Ly::STRIDE;
                        float kr[RPL], qr[RPL];
                        load_rows<RPL>(s_k + ro, kr);
                        if (GATE) {
                            float ar[RPL];
                            load_rows<RPL>(s_a + ro, ar);
#pragma unroll
                            for (int i = 0; i < RPL; i++) S[i] = mul2(S[i], make_float2(ar[i], ar[i]));
                        }
                        float2 p0 = make_float2(0.f, 0.f), p1 = p0;
#pragma unroll
                        for (int i = 0; i < RPL; i += 2) {
                            p0 = fma2(S[i], make_float2(kr[i], kr[i]), p0);
                            p1 = fma2(S[i + 1], make_float2(kr[i + 1], kr[i + 1]), p1);
                        }
                        const float2 p = rowgroup_sum(make_float2(p0.x + p1.x, p0.y + p1.y));
                        const float2 v2 = *reinterpret_cast<const float2*>(s_v + t * kCols + c);
                        const float b = s_b[t];
                        const float2 u = make_float2(b * (v2.x - p.x), b * (v2.y - p.y));
                        load_rows<RPL>(s_q + ro, qr);
                        float2 o0 = make_float2(0.f, 0.f), o1 = o0;
#pragma unroll
                        for (int i = 0; i < RPL; i += 2) {
                            S[i] = fma2(make_float2(kr[i], kr[i]), u, S[i]);
                            S[i + 1] = fma2(make_float2(kr[i + 1], kr[i + 1]), u, S[i + 1]);
                            o0 = fma2(make_float2(qr[i], qr[i]), S[i], o0);
                            o1 = fma2(make_float2(qr[i + 1], qr[i + 1]), S[i + 1], o1);
                        }
                        acc[uu] = make_float2(o0.x + o1.x, o0.y + o1.y);
                    }
                }
                const float o = reduce_scatter<kRB>(acc, lane);
                const int tt = h * kRB + tb_l;
                if (tt < n && writer) {
                    const long oi = (bh * L + t0 + tt) * (long)dv + col0 + c + w_l;
                    if (OUT_F32)
                        static_cast<float*>(a.out)[oi] = o;
                    else
                        static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(o);
                }
            }
        }
        if (more) stage(t0 + kTB, sm + ((rnd + 1) & 1) * Ly::BUF);
        __syncthreads();
    }
    if (active && a.final_state) {  // may alias init_state: each lane read its own entries first
        float* fs = a.final_state + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int i = 0; i < RPL; i++) *reinterpret_cast<float2*>(fs + (long)(r0 + i) * dv) = S[i];
    }
}

template <int RPL, bool GATE, bool OUT_F32>
cudaError_t launch_rpl(const DeltaArgs& a, cudaStream_t s) {
    auto kern = gla_delta_kernel<RPL, GATE, OUT_F32>;
    const size_t smem = DeltaLayout<RPL>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((long)a.B * a.H), (unsigned)((a.dv + kCols - 1) / kCols));
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int RPL>
cudaError_t launch_g(const DeltaArgs& a, cudaStream_t s) {
    const bool f32 = a.out_dtype == GLA_DTYPE_F32;
    if (a.log_alpha) return f32 ? launch_rpl<RPL, true, true>(a, s) : launch_rpl<RPL, true, false>(a, s);
    return f32 ? launch_rpl<RPL, false, true>(a, s) : launch_rpl<RPL, false, false>(a, s);
}

}  // namespace

bool delta_supported(int dk, int dv) {
    return (dk == 32 || dk == 64 || dk == 128) && dv >= 16 && dv % 16 == 0;
}

cudaError_t launch_delta(const DeltaArgs& a, cudaStream_t s) {
    if ((long)a.B * a.H == 0 || a.L == 0) return cudaSuccess;
    if (a.dk == 32) return launch_g<2>(a, s);
    if (a.dk == 64) return launch_g<4>(a, s);
    return launch_g<8>(a, s);
}

}  // namespace gla
