// gla_short.cu -- sequences of 1..16 tokens per call, memory-bound.
//
// "linear-attention" blog, Linear attention: with a fixed-size state, new
// tokens need only that state and themselves, and "Attention is recurrent":
// decoding-sized work is bound by memory bandwidth.  "Gated Linear
// Attention", GLA Recurrent Form:  S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T,
// o_t = S_t^T q_t, applied token by token (exactly the chunk form's result).
//
// This is the hand-off from prefill to multi-token decode: the fp32 state of
// one (batch*head) is read into registers once, the L <= 16 tokens are applied
// in order and the state is written back once, so a call costs one pass over
// the state -- the traffic of a single decode step -- for up to 16 tokens.
// Each thread owns one float4 of value columns for kRows consecutive key rows
// (64 floats), so its per-token alpha, k and q come in as float4 shared loads;
// the updates run as packed fp32 pairs.  Each CTA also prefetches the state
// and tokens of the head about one wave of CTAs ahead into L2.  The per-token partial outputs over
// those rows go to shared memory and are summed over the row groups after the
// token loop (one barrier per call).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kRows = 16;     // key rows per thread
constexpr int kMaxTokens = 16;
constexpr int kMaxThreads = 512;

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// d = a * b + c on fp32 pairs (one instruction, two IEEE round-to-nearest results)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ void l2_prefetch(const void* p, int bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <bool GATE>
__global__ void __launch_bounds__(kMaxThreads) gla_prefill_short_kernel(const PrefillArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int dk = a.dk, dv = a.dv, L = a.L;
    const int cols4 = dv >> 2, rows_par = dk / kRows;
    const long bh = blockIdx.x;
    const int tid = threadIdx.x, nthr = blockDim.x;  // nthr == cols4 * rows_par
    float* s_q = sm;                 // [L][dk]
    float* s_k = s_q + L * dk;       // [L][dk]
    float* s_a = s_k + L * dk;       // [L][dk]  alpha = e^{log alpha}
    float* s_v = s_a + L * dk;       // [L][dv]
    float4* s_red = reinterpret_cast<float4*>(s_v + L * dv);  // [L][rows_par][cols4]

    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + bh * L * dk;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + bh * L * dk;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + bh * L * dv;
    // per-channel gate: [L][dk]; per-token gate (GLA_FLAG_SCALAR_GATE): [L], shared by all channels
    const bool scalar_gate = a.flags & GLA_FLAG_SCALAR_GATE;
    // the head pf_dist CTAs ahead: its state and tokens into L2 while this one is processed
    if (tid == 0 && bh + a.pf_dist < (long)a.B * a.H) {
        const long nb = bh + a.pf_dist;
        if (a.init_state) l2_prefetch(a.init_state + nb * (long)dk * dv, dk * dv * 4);
        l2_prefetch(static_cast<const __nv_bfloat16*>(a.q) + nb * L * dk, L * dk * 2);
        l2_prefetch(static_cast<const __nv_bfloat16*>(a.k) + nb * L * dk, L * dk * 2);
        if ((L * dv * 2) % 16 == 0)  // bulk prefetches take 16-byte multiples (dv % 4 == 0 here)
            l2_prefetch(static_cast<const __nv_bfloat16*>(a.v) + nb * L * dv, L * dv * 2);
        if (GATE && !scalar_gate) l2_prefetch(a.log_alpha + nb * L * dk, L * dk * 4);
    }
    for (int i = tid; i < L * dk; i += nthr) {
        s_q[i] = __bfloat162float(q[i]);
        s_k[i] = __bfloat162float(k[i]);
        if (GATE)
            s_a[i] = __expf(scalar_gate ? a.log_alpha[bh * L + i / dk] : a.log_alpha[bh * L * dk + i]);
        else
            s_a[i] = 1.f;
    }
    for (int i = tid; i < L * dv; i += nthr) s_v[i] = __bfloat162float(v[i]);

    // this thread's rows r = rg * kRows + j (consecutive threads: consecutive float4 of a row)
    const int c4 = tid % cols4, rg = tid / cols4;
    const int r0 = rg * kRows;
    float4 S[kRows];
    if (a.init_state) {
        const float4* S0 = reinterpret_cast<const float4*>(a.init_state + bh * (long)dk * dv);
#pragma unroll
        for (int j = 0; j < kRows; j++) S[j] = __ldcs(&S0[(long)(r0 + j) * cols4 + c4]);
    } else {
#pragma unroll
        for (int j = 0; j < kRows; j++) S[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    for (int t = 0; t < L; t++) {
        const float4 vv = reinterpret_cast<const float4*>(s_v + t * dv)[c4];
        const float2 v01 = make_float2(vv.x, vv.y), v23 = make_float2(vv.z, vv.w);
        const float4* q4 = reinterpret_cast<const float4*>(s_q + t * dk + r0);
        const float4* k4 = reinterpret_cast<const float4*>(s_k + t * dk + r0);
        const float4* a4 = reinterpret_cast<const float4*>(s_a + t * dk + r0);
        float2 acc01 = make_float2(0.f, 0.f), acc23 = acc01;
#pragma unroll
        for (int g = 0; g < kRows / 4; g++) {
            const float4 al4 = a4[g], kk4 = k4[g], qq4 = q4[g];
            const float al[4] = {al4.x, al4.y, al4.z, al4.w}, kk[4] = {kk4.x, kk4.y, kk4.z, kk4.w},
                        qq[4] = {qq4.x, qq4.y, qq4.z, qq4.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float4& sj = S[g * 4 + e];
                const float2 al2 = make_float2(al[e], al[e]), kk2 = make_float2(kk[e], kk[e]),
                             qq2 = make_float2(qq[e], qq[e]);
                // S = alpha S + k v^T (the recurrence's order: decay, then write), then o += q S
                const float2 s01 = fma2(al2, make_float2(sj.x, sj.y), mul2(kk2, v01));
                const float2 s23 = fma2(al2, make_float2(sj.z, sj.w), mul2(kk2, v23));
                sj = make_float4(s01.x, s01.y, s23.x, s23.y);
                acc01 = fma2(qq2, s01, acc01);
                acc23 = fma2(qq2, s23, acc23);
            }
        }
        s_red[(t * rows_par + rg) * cols4 + c4] = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
    }
    if (a.final_state) {  // may alias init_state: this CTA read its whole slice above
        float4* Sf = reinterpret_cast<float4*>(a.final_state + bh * (long)dk * dv);
#pragma unroll
        for (int j = 0; j < kRows; j++) __stcs(&Sf[(long)(r0 + j) * cols4 + c4], S[j]);
    }
    __syncthreads();

    for (int idx = tid; idx < L * cols4; idx += nthr) {
        const int t = idx / cols4, cc = idx % cols4;
        float4 o = s_red[(t * rows_par) * cols4 + cc];
        for (int rr = 1; rr < rows_par; rr++) {
            const float4 p = s_red[(t * rows_par + rr) * cols4 + cc];
            o.x += p.x;
            o.y += p.y;
            o.z += p.z;
            o.w += p.w;
        }
        const long oi = (bh * L + t) * (long)cols4 + cc;
        if (a.out_dtype == GLA_DTYPE_F32)
            reinterpret_cast<float4*>(a.out)[oi] = o;
        else
            reinterpret_cast<uint2*>(a.out)[oi] = make_uint2(pack_bf16x2_rn(o.x, o.y), pack_bf16x2_rn(o.z, o.w));
    }
}

size_t short_smem_bytes(const PrefillArgs& a) {
    return (size_t)a.L * (3 * a.dk + a.dv) * sizeof(float) + (size_t)a.L * a.dk * a.dv / 4;
}

}  // namespace

bool prefill_short_supported(const PrefillArgs& a) {
    if (a.L < 1 || a.L > kMaxTokens) return false;
    if (a.in_dtype != GLA_DTYPE_BF16) return false;
    if (a.flags & (GLA_FLAG_FEATURE_ELU1 | GLA_FLAG_NORMALIZE | GLA_FLAG_FORCE_SIMT | GLA_FLAG_FORCE_CHUNK))
        return false;
    if (a.dk % kRows != 0 || a.dv % 4 != 0) return false;
    const long threads = (long)a.dk * a.dv / (4 * kRows);
    if (threads < 32 || threads > kMaxThreads || threads % 32 != 0) return false;
    if ((long)a.B * a.H > 0x7fffffffL) return false;
    return short_smem_bytes(a) <= 227 * 1024;
}

cudaError_t launch_prefill_short(const PrefillArgs& a_in, cudaStream_t s) {
    PrefillArgs a = a_in;
    // prefetch distance: about the CTAs resident at once (two per SM)
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    a.pf_dist = 2 * sms;
    const int threads = a.dk * a.dv / (4 * kRows);
    const size_t smem = short_smem_bytes(a);
    const unsigned grid = (unsigned)((long)a.B * a.H);
    cudaError_t e;
    if (a.log_alpha) {
        e = cudaFuncSetAttribute(gla_prefill_short_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        gla_prefill_short_kernel<true><<<grid, threads, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(gla_prefill_short_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        gla_prefill_short_kernel<false><<<grid, threads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace gla
