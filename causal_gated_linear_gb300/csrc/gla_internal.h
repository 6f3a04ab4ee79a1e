// gla_internal.h -- launcher interfaces shared by the C-ABI layer and the
// kernel translation units (host side only; no torch types).
#pragma once

#include <cuda_runtime.h>
#include <cuda.h>

#include "../../include/gla.h"

namespace gla {

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* init_state;
    const float* init_z;
    void* out;
    float* final_state;
    float* final_z;
    int B, H, L, dk, dv;
    int in_dtype, out_dtype;
    unsigned flags;
    unsigned* err_word;  // device address of the error word
    int pf_dist;         // short-sequence kernel: CTAs ahead whose inputs it prefetches into L2
    unsigned long long wait_ns;  // tensor-core kernel: limit of its pipeline waits
    int test_stall;              // tensor-core kernel: gate role first waits on a barrier nothing completes
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    float* state;
    float* out;
    int B, H, dk, dv;
};

// fp32 SIMT chunk kernel (any dtype; dk <= 256, dv >= 1).
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t s);

// Whether the tensor-core prefill kernel supports this shape/flag combination.
bool prefill_tc_supported(const PrefillArgs& a);

// tcgen05 chunk kernel (bf16 in; dk in {64,128}; dv multiple of 64).
// Returns cudaSuccess, or an error from encoding the tensor maps / launching.
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

// Whether the short-sequence kernel (1..16 tokens, state read and written
// once per call) handles this call.
bool prefill_short_supported(const PrefillArgs& a);
cudaError_t launch_prefill_short(const PrefillArgs& a, cudaStream_t s);

struct DeltaArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    const float* log_alpha;
    const float* init_state;
    void* out;
    float* final_state;
    int B, H, L, dk, dv;
    int out_dtype;
    unsigned flags;              // GLA_FLAG_FORCE_SIMT: the token-by-token kernel
    unsigned* err_word;          // device address of the error word (chunk-form kernel)
    unsigned long long wait_ns;  // limit of the chunk-form kernel's waits
    int only_marked;             // token-by-token kernel: only the CTAs whose block carries the mark
};

// Written by the chunk-form delta rule into the first output element of every
// 64-column block of a head it leaves to the token-by-token kernel (NaN
// patterns that arithmetic does not produce).
constexpr uint16_t kDeltaMarkBf16 = 0xFFC1u;
constexpr uint32_t kDeltaMarkF32 = 0xFFC00001u;

// Delta rule, token by token (one warp per 16 value columns of a head).
bool delta_supported(int dk, int dv);
cudaError_t launch_delta(const DeltaArgs& a, cudaStream_t s);

// Delta rule in chunk form on the tensor cores (d_k = d_v = 128), then the
// token-by-token kernel on the heads it marked.
bool delta_tc_supported(const DeltaArgs& a);
cudaError_t launch_delta_tc(const DeltaArgs& a, cudaStream_t s);

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    const float* log_alpha;
    const float* init_state;
    const float* dfinal;
    float* dq;
    float* dk_out;
    float* dv_out;
    float* dlog_alpha;
    float* dinit;
    int B, H, L, dk, dv;
    int in_dtype;
    unsigned flags;  // GLA_FLAG_SCALAR_GATE: log_alpha and dlog_alpha are [B][H][L]
    unsigned* err_word;          // device address of the error word (chunk-form kernels)
    unsigned long long wait_ns;  // limit of the chunk-form kernels' waits
    int only_marked;             // recurrent kernel: only the CTAs whose block carries kBwdMark
};

// Written by the chunk-form backward into the first dk / dv element of every
// 32-column block of a head it leaves to the recurrent kernel (a NaN pattern
// that arithmetic does not produce).
constexpr uint32_t kBwdMark = 0xFFC00001u;

// Gradients of the recurrence (row CTAs: dq, dk, dlog_alpha, dS_init;
// column CTAs: dv), one launch.
bool bwd_supported(int dk, int dv);
int bwd_blocks(int d);  // CTAs per head along one dimension (row CTAs for dk, column CTAs for dv)
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s);

// Gradients in chunk form on the tensor cores (bf16, d_k = d_v = 128, one gate
// per channel or none): a dq pass, a dk/dv pass, then the recurrent kernel on
// the heads the chunk form marked.
bool bwd_tc_supported(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s);

// Memory-bound decode step.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// Driver entry point for cuTensorMapEncodeTiled (resolved through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

}  // namespace gla
