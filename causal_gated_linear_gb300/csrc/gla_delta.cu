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
// are column-wise given k_n and beta_n), so a warp owns 16 value columns of
// one head for the whole sequence and needs no block-wide synchronisation per
// token: lane (rg, cq) holds rows [rg * RPL, (rg + 1) * RPL) of columns
// [4 cq, 4 cq + 4) (RPL = dk / 8 rows, 4 * RPL fp32 registers), and the two
// reductions over dk per token (the prediction and the output) are three
// butterfly shuffles across the eight row groups.  Tokens are staged in shared
// memory 32 at a time by the whole CTA (4 warps = 64 value columns); rows are
// padded so that the eight row groups' float4 reads fall in distinct banks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kWarps = 4;             // 16 value columns each
constexpr int kCols = 16 * kWarps;    // value columns per CTA
constexpr int kTB = 32;               // tokens staged per round

template <int RPL>
struct DeltaLayout {
    static constexpr int DK = RPL * 8;
    static constexpr int STRIDE = RPL == 4 ? 12 : RPL + 4;  // padded floats per row group
    static constexpr int ROW = 8 * STRIDE;                  // padded floats per token
    __host__ __device__ static constexpr int pidx(int r) { return (r / RPL) * STRIDE + r % RPL; }
    static constexpr size_t bytes = sizeof(float) * (size_t)kTB * (3 * ROW + kCols + 1);
};

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// sum over the eight row groups (lane bits 2..4)
__device__ __forceinline__ float rowgroup_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

template <int RPL, bool GATE, bool OUT_F32>
__global__ void __launch_bounds__(kWarps * 32) gla_delta_kernel(const DeltaArgs a) {
    using Ly = DeltaLayout<RPL>;
    constexpr int DK = Ly::DK;
    extern __shared__ __align__(16) float sm[];
    float* s_q = sm;                        // [kTB][ROW]
    float* s_k = s_q + kTB * Ly::ROW;       // [kTB][ROW]
    float* s_a = s_k + kTB * Ly::ROW;       // [kTB][ROW]  alpha = e^{log alpha}
    float* s_v = s_a + kTB * Ly::ROW;       // [kTB][kCols]
    float* s_b = s_v + kTB * kCols;         // [kTB]

    const int L = a.L, dv = a.dv;
    const long bh = blockIdx.x;
    const int col0 = blockIdx.y * kCols;
    const int ncols = min(kCols, dv - col0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2, cq = lane & 3;
    const int c = warp * 16 + cq * 4;       // this lane's first column within the CTA's block
    const bool active = c < ncols;          // dv is a multiple of 16, so warps are all or nothing
    const int r0 = rg * RPL;

    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + bh * (long)L * DK;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + bh * (long)L * DK;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + bh * (long)L * dv;
    const float* la = GATE ? a.log_alpha + bh * (long)L * DK : nullptr;
    const float* beta = a.beta + bh * (long)L;

    float S[RPL][4];
    if (active && a.init_state) {
        const float* s0 = a.init_state + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int i = 0; i < RPL; i++) {
            const float4 x = *reinterpret_cast<const float4*>(s0 + (long)(r0 + i) * dv);
            S[i][0] = x.x, S[i][1] = x.y, S[i][2] = x.z, S[i][3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < RPL; i++) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
    }

    for (int t0 = 0; t0 < L; t0 += kTB) {
        const int n = min(kTB, L - t0);
        __syncthreads();  // the previous round's tokens are consumed
        for (int idx = threadIdx.x; idx < n * DK; idx += kWarps * 32) {
            const int t = idx / DK, r = idx % DK;
            const long g = (long)(t0 + t) * DK + r;
            const int o = t * Ly::ROW + Ly::pidx(r);
            s_q[o] = __bfloat162float(q[g]);
            s_k[o] = __bfloat162float(k[g]);
            if (GATE) s_a[o] = __expf(la[g]);
        }
        for (int idx = threadIdx.x; idx < n * ncols; idx += kWarps * 32) {
            const int t = idx / ncols, j = idx % ncols;
            s_v[t * kCols + j] = __bfloat162float(v[(long)(t0 + t) * dv + col0 + j]);
        }
        for (int t = threadIdx.x; t < n; t += kWarps * 32) s_b[t] = beta[t0 + t];
        __syncthreads();
        if (!active) continue;
        for (int t = 0; t < n; t++) {
            const float* kt = s_k + t * Ly::ROW + rg * Ly::STRIDE;
            const float* qt = s_q + t * Ly::ROW + rg * Ly::STRIDE;
            const float* at = s_a + t * Ly::ROW + rg * Ly::STRIDE;
            // the gate decays the state before the prediction
            if (GATE) {
#pragma unroll
                for (int i4 = 0; i4 < RPL; i4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(at + i4);
                    const float al[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int e = 0; e < 4; e++)
#pragma unroll
                        for (int j = 0; j < 4; j++) S[i4 + e][j] *= al[e];
                }
            }
            // prediction p = S^T k for this lane's four columns
            float kr[RPL];
#pragma unroll
            for (int i4 = 0; i4 < RPL; i4 += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(kt + i4);
                kr[i4] = k4.x, kr[i4 + 1] = k4.y, kr[i4 + 2] = k4.z, kr[i4 + 3] = k4.w;
            }
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < RPL; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) p[j] = fmaf(S[i][j], kr[i], p[j]);
#pragma unroll
            for (int j = 0; j < 4; j++) p[j] = rowgroup_sum(p[j]);
            // the error, written with strength beta: S += k u^T
            const float4 v4 = *reinterpret_cast<const float4*>(s_v + t * kCols + c);
            const float b = s_b[t];
            const float u[4] = {b * (v4.x - p[0]), b * (v4.y - p[1]), b * (v4.z - p[2]), b * (v4.w - p[3])};
            float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i4 = 0; i4 < RPL; i4 += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(qt + i4);
                const float qr[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; e++)
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        S[i4 + e][j] = fmaf(kr[i4 + e], u[j], S[i4 + e][j]);
                        o[j] = fmaf(qr[e], S[i4 + e][j], o[j]);
                    }
            }
#pragma unroll
            for (int j = 0; j < 4; j++) o[j] = rowgroup_sum(o[j]);
            if (rg == 0) {
                const long oi = (bh * L + t0 + t) * (long)dv + col0 + c;
                if (OUT_F32)
                    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + oi) = make_float4(o[0], o[1], o[2], o[3]);
                else
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) =
                        make_uint2(pack_bf16x2_rn(o[0], o[1]), pack_bf16x2_rn(o[2], o[3]));
            }
        }
    }
    if (active && a.final_state) {  // may alias init_state: each lane read its own entries first
        float* fs = a.final_state + bh * (long)DK * dv + col0 + c;
#pragma unroll
        for (int i = 0; i < RPL; i++)
            *reinterpret_cast<float4*>(fs + (long)(r0 + i) * dv) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
}

template <int RPL, bool GATE, bool OUT_F32>
cudaError_t launch_rpl(const DeltaArgs& a, cudaStream_t s) {
    auto kern = gla_delta_kernel<RPL, GATE, OUT_F32>;
    const size_t smem = DeltaLayout<RPL>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((long)a.B * a.H), (unsigned)((a.dv + kCols - 1) / kCols));
    kern<<<grid, kWarps * 32, smem, s>>>(a);
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
    if (a.dk == 32) return launch_g<4>(a, s);
    if (a.dk == 64) return launch_g<8>(a, s);
    return launch_g<16>(a, s);
}

}  // namespace gla
