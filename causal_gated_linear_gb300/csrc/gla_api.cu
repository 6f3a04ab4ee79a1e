// gla_api.cu -- the C ABI declared in include/gla.h: host-side validation,
// dispatch to the kernels, and the device error word.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {

// Device error record.  [0]: flags (bitwise OR) set by kernels whose bounded
// pipeline waits ran out; [1..3]: details of the first such wait (see
// gla_device_error_detail in gla.h).
__device__ unsigned g_err_word[4];

EncodeTiledFn encode_tiled_fn() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiledFn>(fn);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool sync_check_enabled() {
    const char* e = std::getenv("GLA_SYNC_CHECK");
    return e && e[0] == '1';
}

// Test hooks (see gla_test_set_waits in gla.h): the limit of the prefill
// kernel's pipeline waits, whether its gate role first waits on a barrier that
// nothing completes, and a launch failure injected after validation when
// GLA_TEST_FAIL_LAUNCH=1 is set in the environment.
unsigned long long g_wait_ns = kWaitLimitNs;
int g_stall = 0;

bool launch_failure_injected() {
    const char* e = std::getenv("GLA_TEST_FAIL_LAUNCH");
    return e && e[0] == '1';
}

unsigned* err_word_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned*>(p);
}

int read_and_clear_error(cudaStream_t s) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return GLA_ERR_CUDA;
    unsigned w = 0;
    if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return GLA_ERR_CUDA;
    if (w) {
        const unsigned zero[4] = {0, 0, 0, 0};
        if (cudaMemcpyToSymbol(g_err_word, zero, sizeof(zero)) != cudaSuccess) return GLA_ERR_CUDA;
        return GLA_ERR_TIMEOUT;
    }
    return GLA_OK;
}

int finish(cudaError_t e, cudaStream_t s) {
    if (e != cudaSuccess) return GLA_ERR_CUDA;
    if (sync_check_enabled()) {
        if (cudaGetLastError() != cudaSuccess) return GLA_ERR_CUDA;
        return read_and_clear_error(s);
    }
    return GLA_OK;
}

int validate_prefill(const gla_fwd_args* a) {
    if (!a) return GLA_ERR_INVALID;
    if (a->B < 1 || a->H < 1 || a->L < 0 || a->dk < 1 || a->dv < 1) return GLA_ERR_INVALID;
    if (a->in_dtype != GLA_DTYPE_BF16 && a->in_dtype != GLA_DTYPE_F32) return GLA_ERR_INVALID;
    if (a->out_dtype != GLA_DTYPE_BF16 && a->out_dtype != GLA_DTYPE_F32) return GLA_ERR_INVALID;
    if (a->flags & ~31u) return GLA_ERR_INVALID;
    if (a->L > 0 && (!a->q || !a->k || !a->v || !a->out)) return GLA_ERR_INVALID;
    if (a->chunk != 64) return GLA_ERR_UNSUPPORTED;
    if (a->dk > 256) return GLA_ERR_UNSUPPORTED;
    const void* ptrs[] = {a->q, a->k, a->v, a->log_alpha, a->init_state, a->init_z, a->out, a->final_state,
                          a->final_z};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GLA_ERR_MISALIGNED;
    const size_t BH = (size_t)a->B * a->H, L = (size_t)a->L;
    const size_t es = a->in_dtype == GLA_DTYPE_F32 ? 4 : 2, eo = a->out_dtype == GLA_DTYPE_F32 ? 4 : 2;
    const size_t nq = BH * L * a->dk * es, nv = BH * L * a->dv * es, no = BH * L * a->dv * eo;
    const size_t nla = BH * L * ((a->flags & GLA_FLAG_SCALAR_GATE) ? 1 : a->dk) * 4;
    const size_t ns = BH * a->dk * a->dv * 4, nz = BH * a->dk * 4;
    if (overlaps(a->out, no, a->q, nq) || overlaps(a->out, no, a->k, nq) || overlaps(a->out, no, a->v, nv) ||
        overlaps(a->out, no, a->log_alpha, nla) || overlaps(a->out, no, a->init_state, ns) ||
        overlaps(a->out, no, a->final_state, ns))
        return GLA_ERR_INVALID;
    // final_state may alias init_state exactly, but not partially
    if (a->final_state && a->init_state && a->final_state != a->init_state &&
        overlaps(a->final_state, ns, a->init_state, ns))
        return GLA_ERR_INVALID;
    if (a->final_z && a->init_z && a->final_z != a->init_z && overlaps(a->final_z, nz, a->init_z, nz))
        return GLA_ERR_INVALID;
    return GLA_OK;
}

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" {

int gla_fwd_ex(const gla_fwd_args* a, void* stream) {
    int st = validate_prefill(a);
    if (st != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PrefillArgs pa;
    pa.q = a->q;
    pa.k = a->k;
    pa.v = a->v;
    pa.log_alpha = a->log_alpha;
    pa.init_state = a->init_state;
    pa.init_z = a->init_z;
    pa.out = a->out;
    pa.final_state = a->final_state;
    pa.final_z = a->final_z;
    pa.B = a->B;
    pa.H = a->H;
    pa.L = a->L;
    pa.dk = a->dk;
    pa.dv = a->dv;
    pa.in_dtype = a->in_dtype;
    pa.out_dtype = a->out_dtype;
    pa.flags = a->flags;
    pa.pf_dist = 0;
    pa.wait_ns = g_wait_ns;
    pa.test_stall = g_stall;
    const size_t BH = (size_t)a->B * a->H;
    if (a->L == 0) {
        // no tokens: the final state is the initial one
        cudaError_t e = cudaSuccess;
        const size_t ns = BH * a->dk * a->dv * sizeof(float), nz = BH * a->dk * sizeof(float);
        if (a->final_state && a->final_state != a->init_state)
            e = a->init_state ? cudaMemcpyAsync(a->final_state, a->init_state, ns, cudaMemcpyDeviceToDevice, s)
                              : cudaMemsetAsync(a->final_state, 0, ns, s);
        if (e == cudaSuccess && a->final_z && (a->flags & GLA_FLAG_NORMALIZE) && a->final_z != a->init_z)
            e = a->init_z ? cudaMemcpyAsync(a->final_z, a->init_z, nz, cudaMemcpyDeviceToDevice, s)
                          : cudaMemsetAsync(a->final_z, 0, nz, s);
        return finish(e, s);
    }
    if (launch_failure_injected()) return GLA_ERR_CUDA;
    pa.err_word = err_word_ptr();
    if (!pa.err_word) return GLA_ERR_CUDA;
    cudaError_t e;
    if (prefill_short_supported(pa)) {
        e = launch_prefill_short(pa, s);
    } else if (prefill_tc_supported(pa)) {
        e = launch_prefill_tc(pa, s);
    } else {
        if (BH > 65535) return GLA_ERR_UNSUPPORTED;
        e = launch_prefill_simt(pa, s);
    }
    return finish(e, s);
}

int gla_fwd_host(const gla_fwd_args* host, const gla_fwd_args* dev, int groups, void* copy_in, void* compute,
                 void* copy_out) {
    if (!host || !dev || groups < 1) return GLA_ERR_INVALID;
    int st = validate_prefill(dev);
    if (st != GLA_OK) return st;
    if (host->B != dev->B || host->H != dev->H || host->L != dev->L || host->dk != dev->dk || host->dv != dev->dv ||
        host->chunk != dev->chunk || host->in_dtype != dev->in_dtype || host->out_dtype != dev->out_dtype ||
        host->flags != dev->flags)
        return GLA_ERR_INVALID;
    // every buffer is given on both sides or on neither
    const void* hp[] = {host->q, host->k, host->v, host->log_alpha, host->init_state, host->init_z,
                        host->out, host->final_state, host->final_z};
    const void* dp[] = {dev->q, dev->k, dev->v, dev->log_alpha, dev->init_state, dev->init_z,
                        dev->out, dev->final_state, dev->final_z};
    for (int i = 0; i < 9; i++)
        if ((hp[i] == nullptr) != (dp[i] == nullptr)) return GLA_ERR_INVALID;
    if (dev->final_state && dev->final_state == dev->init_state) return GLA_ERR_INVALID;  // staged separately
    if (dev->final_z && dev->final_z == dev->init_z) return GLA_ERR_INVALID;
    cudaStream_t s_in = static_cast<cudaStream_t>(copy_in), s_c = static_cast<cudaStream_t>(compute),
                 s_out = static_cast<cudaStream_t>(copy_out);
    const long BH = (long)dev->B * dev->H;
    const size_t L = (size_t)dev->L;
    const size_t es = dev->in_dtype == GLA_DTYPE_F32 ? 4 : 2, eo = dev->out_dtype == GLA_DTYPE_F32 ? 4 : 2;
    const bool normz = dev->flags & GLA_FLAG_NORMALIZE;
    // bytes per head of each buffer, in the order of hp / dp
    const size_t per[] = {L * dev->dk * es, L * dev->dk * es, L * dev->dv * es,
                          L * ((dev->flags & GLA_FLAG_SCALAR_GATE) ? 1 : dev->dk) * 4, (size_t)dev->dk * dev->dv * 4,
                          normz ? (size_t)dev->dk * 4 : 0, L * dev->dv * eo, (size_t)dev->dk * dev->dv * 4,
                          normz ? (size_t)dev->dk * 4 : 0};
    // group boundaries fall on multiples of `gran` heads, so that every slice of
    // every buffer starts 16-byte aligned (a head's bytes are a multiple of 2)
    long gran = 1;
    for (size_t b : per) {
        long need = 1;
        while (b > 0 && (b * need) % 16 != 0) need *= 2;
        if (need > gran) gran = need;
    }
    const long units = (BH + gran - 1) / gran;
    const int G = (int)(groups < units ? groups : units);
    cudaEvent_t start_c, start_out;
    if (cudaEventCreateWithFlags(&start_c, cudaEventDisableTiming) != cudaSuccess) return GLA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&start_out, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(start_c);
        return GLA_ERR_CUDA;
    }
    // inputs are overwritten only after earlier kernels on `compute` have read them, outputs
    // only after earlier copies on `copy_out` have read them
    cudaError_t e = cudaEventRecord(start_c, s_c);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, start_c, 0);
    if (e == cudaSuccess) e = cudaEventRecord(start_out, s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_c, start_out, 0);
    cudaEventDestroy(start_c);
    cudaEventDestroy(start_out);
    if (e != cudaSuccess) return GLA_ERR_CUDA;
    for (int g = 0; g < G; g++) {
        const long u0 = units * g / G, u1 = units * (g + 1) / G;
        const long h0 = u0 * gran < BH ? u0 * gran : BH, h1 = u1 * gran < BH ? u1 * gran : BH, nh = h1 - h0;
        const void* hs[9];
        void* ds[9];
        for (int i = 0; i < 9; i++) {
            hs[i] = hp[i] ? static_cast<const char*>(hp[i]) + h0 * per[i] : nullptr;
            ds[i] = dp[i] ? const_cast<char*>(static_cast<const char*>(dp[i])) + h0 * per[i] : nullptr;
        }
        for (int i = 0; i < 6; i++)
            if (ds[i] && nh * per[i] > 0 &&
                cudaMemcpyAsync(ds[i], hs[i], nh * per[i], cudaMemcpyHostToDevice, s_in) != cudaSuccess)
                return GLA_ERR_CUDA;
        cudaEvent_t landed, done;
        if (cudaEventCreateWithFlags(&landed, cudaEventDisableTiming) != cudaSuccess) return GLA_ERR_CUDA;
        e = cudaEventRecord(landed, s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_c, landed, 0);
        cudaEventDestroy(landed);
        if (e != cudaSuccess) return GLA_ERR_CUDA;
        gla_fwd_args ga = *dev;  // the group's heads as one batch of nh heads
        ga.B = 1;
        ga.H = (int)nh;
        ga.q = ds[0], ga.k = ds[1], ga.v = ds[2];
        ga.log_alpha = static_cast<const float*>(ds[3]);
        ga.init_state = static_cast<const float*>(ds[4]);
        ga.init_z = static_cast<const float*>(ds[5]);
        ga.out = ds[6];
        ga.final_state = static_cast<float*>(ds[7]);
        ga.final_z = static_cast<float*>(ds[8]);
        st = gla_fwd_ex(&ga, s_c);
        if (st != GLA_OK) return st;
        if (cudaEventCreateWithFlags(&done, cudaEventDisableTiming) != cudaSuccess) return GLA_ERR_CUDA;
        e = cudaEventRecord(done, s_c);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, done, 0);
        cudaEventDestroy(done);
        if (e != cudaSuccess) return GLA_ERR_CUDA;
        for (int i = 6; i < 9; i++)
            if (ds[i] && nh * per[i] > 0 &&
                cudaMemcpyAsync(const_cast<void*>(hs[i]), ds[i], nh * per[i], cudaMemcpyDeviceToHost, s_out) !=
                    cudaSuccess)
                return GLA_ERR_CUDA;
    }
    return finish(cudaSuccess, s_out);
}

int gla_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* init_state, void* out,
            float* final_state, int B, int H, int L, int dk, int dv, int chunk, void* stream) {
    gla_fwd_args a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.log_alpha = log_alpha;
    a.init_state = init_state;
    a.out = out;
    a.final_state = final_state;
    a.B = B;
    a.H = H;
    a.L = L;
    a.dk = dk;
    a.dv = dv;
    a.chunk = chunk;
    a.in_dtype = GLA_DTYPE_BF16;
    a.out_dtype = GLA_DTYPE_BF16;
    a.flags = 0;
    return gla_fwd_ex(&a, stream);
}

int gla_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, float* state, float* out,
                    int B, int H, int dk, int dv, void* stream) {
    if (B < 1 || H < 1 || dk < 1 || dv < 1) return GLA_ERR_INVALID;
    if (!q || !k || !v || !state || !out) return GLA_ERR_INVALID;
    if (dv % 4 != 0 || dv > 512 || dk > 512) return GLA_ERR_UNSUPPORTED;
    if ((size_t)B * H > 0x7fffffffu) return GLA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, log_alpha, state, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GLA_ERR_MISALIGNED;
    const size_t BH = (size_t)B * H;
    const size_t no = BH * dv * 4;
    if (overlaps(out, no, state, BH * dk * dv * 4) || overlaps(out, no, q, BH * dk * 2) ||
        overlaps(out, no, k, BH * dk * 2) || overlaps(out, no, v, BH * dv * 2) ||
        overlaps(out, no, log_alpha, BH * dk * 4))
        return GLA_ERR_INVALID;
    DecodeArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.log_alpha = log_alpha;
    a.state = state;
    a.out = out;
    a.B = B;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_failure_injected()) return GLA_ERR_CUDA;
    return finish(launch_decode(a, s), s);
}

int gla_delta_fwd_ex(const void* q, const void* k, const void* v, const float* beta, const float* log_alpha,
                     const float* init_state, void* out, float* final_state, int B, int H, int L, int dk, int dv,
                     int out_dtype, unsigned flags, void* stream) {
    if (B < 1 || H < 1 || L < 0 || dk < 1 || dv < 1) return GLA_ERR_INVALID;
    if (out_dtype != GLA_DTYPE_BF16 && out_dtype != GLA_DTYPE_F32) return GLA_ERR_INVALID;
    if (flags & ~(unsigned)GLA_FLAG_FORCE_SIMT) return GLA_ERR_INVALID;
    if (L > 0 && (!q || !k || !v || !beta || !out)) return GLA_ERR_INVALID;
    if (!delta_supported(dk, dv)) return GLA_ERR_UNSUPPORTED;
    if ((size_t)B * H > 0x7fffffffu || (dv + 63) / 64 > 65535) return GLA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, beta, log_alpha, init_state, out, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GLA_ERR_MISALIGNED;
    const size_t BH = (size_t)B * H, Ls = (size_t)L;
    const size_t no = BH * Ls * dv * (out_dtype == GLA_DTYPE_F32 ? 4 : 2), ns = BH * dk * dv * 4;
    if (overlaps(out, no, q, BH * Ls * dk * 2) || overlaps(out, no, k, BH * Ls * dk * 2) ||
        overlaps(out, no, v, BH * Ls * dv * 2) || overlaps(out, no, beta, BH * Ls * 4) ||
        overlaps(out, no, log_alpha, BH * Ls * dk * 4) || overlaps(out, no, init_state, ns) ||
        overlaps(out, no, final_state, ns))
        return GLA_ERR_INVALID;
    if (final_state && init_state && final_state != init_state && overlaps(final_state, ns, init_state, ns))
        return GLA_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L == 0) {
        cudaError_t e = cudaSuccess;
        if (final_state && final_state != init_state)
            e = init_state ? cudaMemcpyAsync(final_state, init_state, ns, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(final_state, 0, ns, s);
        return finish(e, s);
    }
    DeltaArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.beta = beta;
    a.log_alpha = log_alpha;
    a.init_state = init_state;
    a.out = out;
    a.final_state = final_state;
    a.B = B;
    a.H = H;
    a.L = L;
    a.dk = dk;
    a.dv = dv;
    a.out_dtype = out_dtype;
    a.flags = flags;
    a.err_word = nullptr;
    a.wait_ns = g_wait_ns;
    a.only_marked = 0;
    if (launch_failure_injected()) return GLA_ERR_CUDA;
    if (delta_tc_supported(a)) {
        a.err_word = err_word_ptr();
        if (!a.err_word) return GLA_ERR_CUDA;
        return finish(launch_delta_tc(a, s), s);
    }
    return finish(launch_delta(a, s), s);
}

int gla_delta_fwd(const void* q, const void* k, const void* v, const float* beta, const float* log_alpha,
                  const float* init_state, void* out, float* final_state, int B, int H, int L, int dk, int dv,
                  int out_dtype, void* stream) {
    return gla_delta_fwd_ex(q, k, v, beta, log_alpha, init_state, out, final_state, B, H, L, dk, dv, out_dtype, 0u,
                            stream);
}

int gla_bwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* init_state,
            const void* dout, const float* dfinal, float* dq, float* dk_out, float* dv_out, float* dlog_alpha,
            float* dinit, int B, int H, int L, int dk, int dv, int in_dtype, unsigned flags, void* stream) {
    if (B < 1 || H < 1 || L < 0 || dk < 1 || dv < 1) return GLA_ERR_INVALID;
    if (in_dtype != GLA_DTYPE_BF16 && in_dtype != GLA_DTYPE_F32) return GLA_ERR_INVALID;
    if (flags & ~(unsigned)(GLA_FLAG_SCALAR_GATE | GLA_FLAG_FORCE_SIMT)) return GLA_ERR_INVALID;
    const bool scalar = flags & GLA_FLAG_SCALAR_GATE;
    if (L > 0 && (!q || !k || !v || !dout || !dq || !dk_out || !dv_out)) return GLA_ERR_INVALID;
    if (dlog_alpha && !log_alpha) return GLA_ERR_INVALID;
    if (!bwd_supported(dk, dv)) return GLA_ERR_UNSUPPORTED;
    if ((size_t)B * H * (bwd_blocks(dk) + bwd_blocks(dv)) > 0x7fffffffu) return GLA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, log_alpha, init_state, dout, dfinal, dq, dk_out, dv_out, dlog_alpha, dinit};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GLA_ERR_MISALIGNED;
    const size_t BH = (size_t)B * H, Ls = (size_t)L, es = in_dtype == GLA_DTYPE_F32 ? 4 : 2;
    const size_t nk = BH * Ls * dk, nv = BH * Ls * dv, ns = BH * dk * dv * 4, nla = scalar ? BH * Ls : nk;
    const void* in_p[] = {q, k, v, dout, log_alpha, init_state, dfinal};
    const size_t in_n[] = {nk * es, nk * es, nv * es, nv * es, nla * 4, ns, ns};
    const void* out_p[] = {dq, dk_out, dv_out, dlog_alpha, dinit};
    const size_t out_n[] = {nk * 4, nk * 4, nv * 4, nla * 4, ns};
    for (int o = 0; o < 5; o++) {
        for (int i = 0; i < 7; i++)
            if (overlaps(out_p[o], out_n[o], in_p[i], in_n[i])) return GLA_ERR_INVALID;
        for (int p = 0; p < o; p++)
            if (overlaps(out_p[o], out_n[o], out_p[p], out_n[p])) return GLA_ERR_INVALID;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L == 0) {
        cudaError_t e = cudaSuccess;
        if (dinit)
            e = dfinal ? cudaMemcpyAsync(dinit, dfinal, ns, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(dinit, 0, ns, s);
        return finish(e, s);
    }
    BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.dout = dout;
    a.log_alpha = log_alpha;
    a.init_state = init_state;
    a.dfinal = dfinal;
    a.dq = dq;
    a.dk_out = dk_out;
    a.dv_out = dv_out;
    a.dlog_alpha = dlog_alpha;
    a.dinit = dinit;
    a.B = B;
    a.H = H;
    a.L = L;
    a.dk = dk;
    a.dv = dv;
    a.in_dtype = in_dtype;
    a.flags = flags;
    a.err_word = nullptr;
    a.wait_ns = g_wait_ns;
    a.only_marked = 0;
    if (launch_failure_injected()) return GLA_ERR_CUDA;
    // a per-token gate's gradient is accumulated across the row blocks of a head
    if (bwd_tc_supported(a)) {
        a.err_word = err_word_ptr();
        if (!a.err_word) return GLA_ERR_CUDA;
        return finish(launch_bwd_tc(a, s), s);
    }
    if (scalar && dlog_alpha && cudaMemsetAsync(dlog_alpha, 0, nla * 4, s) != cudaSuccess) return GLA_ERR_CUDA;
    return finish(launch_bwd(a, s), s);
}

int gla_device_error(void* stream) { return read_and_clear_error(static_cast<cudaStream_t>(stream)); }

int gla_device_error_detail(void* stream, unsigned* detail4) {
    if (!detail4) return GLA_ERR_INVALID;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GLA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(detail4, g_err_word, 4 * sizeof(unsigned)) != cudaSuccess) return GLA_ERR_CUDA;
    return GLA_OK;
}

const char* gla_status_string(int status) {
    switch (status) {
        case GLA_OK: return "GLA_OK";
        case GLA_ERR_INVALID: return "GLA_ERR_INVALID";
        case GLA_ERR_UNSUPPORTED: return "GLA_ERR_UNSUPPORTED";
        case GLA_ERR_MISALIGNED: return "GLA_ERR_MISALIGNED";
        case GLA_ERR_CUDA: return "GLA_ERR_CUDA";
        case GLA_ERR_TIMEOUT: return "GLA_ERR_TIMEOUT";
        default: return "GLA_ERR_UNKNOWN";
    }
}

int gla_test_set_waits(unsigned long long limit_ns, int stall) {
    g_wait_ns = limit_ns ? limit_ns : kWaitLimitNs;
    g_stall = stall ? 1 : 0;
    return GLA_OK;
}

const char* gla_version(void) { return "gla-gb300 0.2.0 (sm_103a)"; }

}  // extern "C"
