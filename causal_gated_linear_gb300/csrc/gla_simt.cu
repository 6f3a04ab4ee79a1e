// gla_simt.cu -- exact-fp32 SIMT chunk kernel.
//
// Evaluates the gated recurrence ("Gated Linear Attention", GLA Recurrent
// Form) in the chunk-wise block-parallel form ("Gated Linear Attention",
// Chunk-Wise Block-Parallel) with plain fp32 FFMA and no tensor cores, so
// that an fp32 configuration can be held to a 1e-5 relative error.  For a
// token block with b_t = inclusive cumsum of log alpha from the block start:
//   o_t = (q_t * e^{b_t})^T S_prev + sum_{i<=t} [sum_d q_td k_id e^{b_td - b_id}] v_i
//   S   = Diag(e^{b_last}) S_prev + sum_i (k_i * e^{b_last - b_i}) v_i^T
// Every exponent is <= 0 (log alpha <= 0), so no intermediate can overflow
// whatever the gate values; the intra-block decay is evaluated per (t, i, d)
// rather than factored, which costs exps but keeps this kernel a robust
// reference-grade GPU path for any shape.  The factors of the inter-block
// term and of the state update (q_t e^{b_t}, k_i e^{b_last - b_i}) are formed
// once per block; the per-pair weights use the fast hardware exponential
// (arguments all <= 0), well inside the fp32 parity bar.
//
// Grid: (value-column tiles of kDVT, B*H).  Block: 256 threads.  Each CTA
// keeps its d_k x kDVT slice of S (plus the normaliser column) in shared
// memory for the whole sequence.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kThreads = 256;
constexpr int kDVT = 32;  // value columns per CTA

template <typename T>
__device__ __forceinline__ float ld_in(const T* p, long i);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p, long i) {
    return p[i];
}
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, long i) {
    return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st_out(T* p, long i, float x);
template <>
__device__ __forceinline__ void st_out<float>(float* p, long i, float x) {
    p[i] = x;
}
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, long i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float phi_elu1_exact(float x) { return x > 0.f ? x + 1.f : expf(x); }

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) gla_prefill_simt_kernel(PrefillArgs a, int TB) {
    extern __shared__ float sm[];
    const int dk = a.dk, dv = a.dv, L = a.L;
    const bool elu = a.flags & GLA_FLAG_FEATURE_ELU1;
    const bool norm = a.flags & GLA_FLAG_NORMALIZE;
    const int NC = kDVT + 1;  // local value columns (+ normaliser)
    // per-token rows of the [TB][dk] tables are padded to DKP = dk + 1 floats: the pair loop
    // reads column d of consecutive rows across a warp, which an unpadded stride of dk
    // (a multiple of 32 words) would put in one shared-memory bank
    const int DKP = dk + 1;
    float* qf = sm;                  // [TB][DKP]
    float* kf = qf + TB * DKP;       // [TB][DKP]
    float* bb = kf + TB * DKP;       // [TB][DKP] cumsum of log alpha
    float* vv = bb + TB * DKP;       // [TB][NC]
    float* S = vv + TB * NC;         // [dk][NC]
    float* A = S + dk * NC;          // [TB][TB]
    float* os = A + TB * TB;         // [TB][NC]
    float* qe = os + TB * NC;        // [TB][DKP] q_t e^{b_t}
    float* kh = qe + TB * DKP;       // [TB][DKP] k_i e^{b_last - b_i}
    float* gl = kh + TB * DKP;       // [dk] e^{b_last}

    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * kDVT;
    const long bh = blockIdx.y;
    const TI* q = static_cast<const TI*>(a.q) + bh * (long)L * dk;
    const TI* k = static_cast<const TI*>(a.k) + bh * (long)L * dk;
    const TI* v = static_cast<const TI*>(a.v) + bh * (long)L * dv;
    // per-channel gate: [L][dk]; per-token gate (GLA_FLAG_SCALAR_GATE): [L], shared by all channels
    const bool scalar_gate = a.flags & GLA_FLAG_SCALAR_GATE;
    const long la_t = scalar_gate ? 1 : dk, la_d = scalar_gate ? 0 : 1;
    const float* la = a.log_alpha ? a.log_alpha + bh * (long)L * la_t : nullptr;
    TO* out = static_cast<TO*>(a.out) + bh * (long)L * dv;

    for (int idx = tid; idx < dk * NC; idx += kThreads) {
        int d = idx / NC, jj = idx % NC;
        float s0 = 0.f;
        if (jj < kDVT) {
            if (a.init_state && j0 + jj < dv) s0 = a.init_state[bh * dk * dv + (long)d * dv + j0 + jj];
        } else if (norm && a.init_z) {
            s0 = a.init_z[bh * dk + d];
        }
        S[idx] = s0;
    }
    __syncthreads();

    for (int t0 = 0; t0 < L; t0 += TB) {
        const int n = min(TB, L - t0);
        for (int idx = tid; idx < TB * dk; idx += kThreads) {
            int t = idx / dk, d = idx % dk;
            float xq = 0.f, xk = 0.f, xl = 0.f;
            if (t < n) {
                long g = (long)(t0 + t) * dk + d;
                xq = ld_in(q, g);
                xk = ld_in(k, g);
                if (elu) {
                    xq = phi_elu1_exact(xq);
                    xk = phi_elu1_exact(xk);
                }
                if (la) xl = la[(long)(t0 + t) * la_t + d * la_d];
            }
            qf[t * DKP + d] = xq;
            kf[t * DKP + d] = xk;
            bb[t * DKP + d] = xl;
        }
        for (int idx = tid; idx < TB * NC; idx += kThreads) {
            int t = idx / NC, jj = idx % NC;
            float x = 0.f;
            if (t < n) {
                if (jj < kDVT) {
                    if (j0 + jj < dv) x = ld_in(v, (long)(t0 + t) * dv + j0 + jj);
                } else if (norm) {
                    x = 1.f;
                }
            }
            vv[idx] = x;
        }
        __syncthreads();
        // inclusive cumsum of log alpha per channel (padding tokens carry 0)
        for (int d = tid; d < dk; d += kThreads) {
            float run = 0.f;
            for (int t = 0; t < TB; t++) {
                run += bb[t * DKP + d];
                bb[t * DKP + d] = run;
            }
            gl[d] = expf(run);
        }
        __syncthreads();
        // factors of the inter-block term and of the state update (exponents <= 0)
        for (int idx = tid; idx < TB * dk; idx += kThreads) {
            const int t = idx / dk, d = idx % dk, o = t * DKP + d;
            qe[o] = qf[o] * expf(bb[o]);
            kh[o] = kf[o] * expf(bb[(TB - 1) * DKP + d] - bb[o]);
        }
        // intra-block scores with the exact decay weight of every pair
        for (int idx = tid; idx < TB * TB; idx += kThreads) {
            int t = idx / TB, i = idx % TB;
            float acc = 0.f;
            if (i <= t) {
                for (int d = 0; d < dk; d++)
                    acc = fmaf(qf[t * DKP + d] * kf[i * DKP + d], __expf(bb[t * DKP + d] - bb[i * DKP + d]), acc);
            }
            A[idx] = acc;
        }
        __syncthreads();
        // outputs: inter-block (decayed state) + intra-block
        for (int idx = tid; idx < TB * NC; idx += kThreads) {
            int t = idx / NC, jj = idx % NC;
            float acc = 0.f;
            for (int d = 0; d < dk; d++) acc = fmaf(qe[t * DKP + d], S[d * NC + jj], acc);
            for (int i = 0; i <= t; i++) acc = fmaf(A[t * TB + i], vv[i * NC + jj], acc);
            os[idx] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < TB * kDVT; idx += kThreads) {
            int t = idx / kDVT, jj = idx % kDVT;
            if (t < n && j0 + jj < dv) {
                float o = os[t * NC + jj];
                if (norm) o = o / os[t * NC + kDVT];
                st_out(out, (long)(t0 + t) * dv + j0 + jj, o);
            }
        }
        // state update (every column incl. the normaliser)
        for (int idx = tid; idx < dk * NC; idx += kThreads) {
            int d = idx / NC, jj = idx % NC;
            float acc = gl[d] * S[idx];
            for (int i = 0; i < TB; i++) acc = fmaf(kh[i * DKP + d], vv[i * NC + jj], acc);
            S[idx] = acc;
        }
        __syncthreads();
    }

    for (int idx = tid; idx < dk * NC; idx += kThreads) {
        int d = idx / NC, jj = idx % NC;
        if (jj < kDVT) {
            if (a.final_state && j0 + jj < dv) a.final_state[bh * dk * dv + (long)d * dv + j0 + jj] = S[idx];
        } else if (norm && a.final_z && blockIdx.x == 0) {
            a.final_z[bh * dk + d] = S[idx];
        }
    }
}

size_t simt_smem_bytes(int dk, int TB) {
    const int NC = kDVT + 1;
    return sizeof(float) * (size_t)(5 * TB * (dk + 1) + TB * NC + dk * NC + TB * TB + TB * NC + dk);
}

template <typename TI, typename TO>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
    const int TB = a.dk <= 128 ? 64 : 32;
    size_t smem = simt_smem_bytes(a.dk, TB);
    auto kern = gla_prefill_simt_kernel<TI, TO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.dv + kDVT - 1) / kDVT, a.B * a.H);
    kern<<<grid, kThreads, smem, s>>>(a, TB);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t s) {
    const bool f32in = a.in_dtype == GLA_DTYPE_F32;
    const bool f32out = a.out_dtype == GLA_DTYPE_F32;
    if (f32in && f32out) return launch_t<float, float>(a, s);
    if (f32in) return launch_t<float, __nv_bfloat16>(a, s);
    if (f32out) return launch_t<__nv_bfloat16, float>(a, s);
    return launch_t<__nv_bfloat16, __nv_bfloat16>(a, s);
}

}  // namespace gla
