// gla_decode.cu -- one recurrent step per (sequence, head), memory-bound.
//
// "linear-attention" blog, Linear attention: with a fixed-size state, token
// n needs only (S_{n-1}, q_n, k_n, v_n); "Attention is recurrent": decoding
// is bound by memory bandwidth.  Gate from "Gated Linear Attention", GLA
// Recurrent Form:  S <- Diag(alpha) S + k v^T  (in place),  o = S^T q.
//
// The fp32 state is streamed exactly once in and once out with 128-bit
// accesses: a CTA owns one (sequence, head); each thread owns one float4 of
// value columns for a stripe of key rows, updates it, writes it back and
// accumulates q_i * S'_i; partial sums over rows are reduced in shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxDk = 512;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) gla_decode_kernel(DecodeArgs a, int pf_dist) {
    __shared__ float s_q[kMaxDk], s_k[kMaxDk], s_a[kMaxDk];
    __shared__ float4 s_red[kThreads];
    const int dk = a.dk, dv = a.dv;
    const long hs = blockIdx.x;
    const int tid = threadIdx.x;
    // the state pf_dist CTAs ahead into L2 while this one streams (16-byte multiples only)
    if (tid == 0 && hs + pf_dist < (long)gridDim.x && (dk * dv) % 4 == 0) {
        const float* nxt = a.state + (hs + pf_dist) * (long)dk * dv;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nxt), "r"(dk * dv * 4) : "memory");
    }
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + hs * dk;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k) + hs * dk;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v) + hs * dv;
    for (int i = tid; i < dk; i += kThreads) {
        s_q[i] = __bfloat162float(q[i]);
        s_k[i] = __bfloat162float(k[i]);
        s_a[i] = a.log_alpha ? __expf(a.log_alpha[hs * dk + i]) : 1.f;
    }
    __syncthreads();

    const int cols4 = dv >> 2;            // float4 columns per row
    const int rows_par = kThreads / cols4; // rows processed concurrently
    const int c4 = tid % cols4;
    const int r0 = tid / cols4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 < rows_par) {
        float4 vv;
        {
            const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(v) + 2 * c4;
            float2 a0 = __bfloat1622float2(v2[0]);
            float2 a1 = __bfloat1622float2(v2[1]);
            vv = make_float4(a0.x, a0.y, a1.x, a1.y);
        }
        float4* S = reinterpret_cast<float4*>(a.state + hs * (long)dk * dv);
        int r = r0;
        for (; r + (kUnroll - 1) * rows_par < dk; r += kUnroll * rows_par) {
            float4 s[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) s[u] = __ldcs(&S[(long)(r + u * rows_par) * cols4 + c4]);
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                const int row = r + u * rows_par;
                const float al = s_a[row], kk = s_k[row], qq = s_q[row];
                s[u].x = fmaf(al, s[u].x, kk * vv.x);
                s[u].y = fmaf(al, s[u].y, kk * vv.y);
                s[u].z = fmaf(al, s[u].z, kk * vv.z);
                s[u].w = fmaf(al, s[u].w, kk * vv.w);
                __stcs(&S[(long)row * cols4 + c4], s[u]);
                acc.x = fmaf(qq, s[u].x, acc.x);
                acc.y = fmaf(qq, s[u].y, acc.y);
                acc.z = fmaf(qq, s[u].z, acc.z);
                acc.w = fmaf(qq, s[u].w, acc.w);
            }
        }
        for (; r < dk; r += rows_par) {
            float4 s = __ldcs(&S[(long)r * cols4 + c4]);
            const float al = s_a[r], kk = s_k[r], qq = s_q[r];
            s.x = fmaf(al, s.x, kk * vv.x);
            s.y = fmaf(al, s.y, kk * vv.y);
            s.z = fmaf(al, s.z, kk * vv.z);
            s.w = fmaf(al, s.w, kk * vv.w);
            __stcs(&S[(long)r * cols4 + c4], s);
            acc.x = fmaf(qq, s.x, acc.x);
            acc.y = fmaf(qq, s.y, acc.y);
            acc.z = fmaf(qq, s.z, acc.z);
            acc.w = fmaf(qq, s.w, acc.w);
        }
    }
    s_red[tid] = acc;
    __syncthreads();
    if (tid < cols4) {
        float4 o = s_red[tid];
        for (int rr = 1; rr < rows_par; rr++) {
            float4 p = s_red[rr * cols4 + tid];
            o.x += p.x;
            o.y += p.y;
            o.z += p.z;
            o.w += p.w;
        }
        reinterpret_cast<float4*>(a.out + hs * (long)dv)[tid] = o;
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    const long n = (long)a.B * a.H;
    if (n == 0) return cudaSuccess;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    gla_decode_kernel<<<dim3((unsigned)n), kThreads, 0, s>>>(a, 3 * sms);  // about the CTAs resident at once
    return cudaGetLastError();
}

}  // namespace gla
