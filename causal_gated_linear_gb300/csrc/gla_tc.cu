// gla_tc.cu -- tcgen05 / TMEM / TMA chunk-wise prefill kernel for sm_103a.
//
// Method ("Gated Linear Attention", GLA Recurrent Form and Chunk-Wise
// Block-Parallel): S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t,
// evaluated 64 tokens at a time.  Unrolling the recurrence over one chunk
// ("linear-attention" blog, Gated linear attention: a write at i reaches t
// weighted by the product of alpha over (i, t]) and writing b_t for the
// inclusive cumsum of log alpha from the chunk start, b_C for its last value:
//   Qh_t = q_t * e^{b_t}              (<= 1 factor)
//   Kh_i = k_i * e^{-b_i}             (>= 1 factor, at most e^{-b_C})
//   o_t  = Qh_t^T S_prev + sum_{i<=t} (Qh_t . Kh_i) v_i    (inter + intra)
//   S    = Diag(e^{b_C}) (S_prev + Kh^T V)
// which is exactly the recurrence, since (Qh_t . Kh_i) carries e^{b_t - b_i}.
// The output product reads the state from before the chunk, so it can start as
// soon as the chunk's factors are written; the state update is off its path.
//
// One CTA owns one (batch*head, DVT-column slice of d_v) for the whole
// sequence (DVT = 64 or 128, chosen by the host so that enough CTAs exist to
// cover the GPU).  The state is kept TRANSPOSED in tensor memory, S^T (lane =
// value column j, column = key channel d, fp32), so that every state/output
// product has M = DVT:
//   MMA_A   A[t][i] = Qh Kh^T          M=128 (rows 64..127 unused), N=64, K=dk
//   MMA_dS  dS^T    = V^T Kh           M=DVT, N=dk, K=64  (V, Kh MN-major; own buffer)
//   MMA_Oi  O^T     = S^T_bf16 Qh^T    M=DVT, N=64, K=dk  (A operand from TMEM)
//   MMA_Oa  O^T    += V^T P^T          M=DVT, N=64, K=64  (P = tril(A) in bf16)
// The state warps form S = Diag(e^{b_C}) (S + dS) in fp32 (in TMEM for the
// 128-column tile, in their registers for the 64-column tile) and write its
// bf16 copy into TMEM for the next chunk's MMA_Oi; no state ever leaves the
// chip between chunks.  With M = 64 the accumulator rows live in TMEM lanes
// 16q + r -> lane 32q + r (r < 16) of each 32-lane quarter q.
//
// Warp roles (24 warps): 0-7 gate (cumsum with a cross-warp segment
// exchange, factors written in place over the TMA-landed q/k tiles), 8-15
// state, 16-19 output (TMEM -> shared staging -> TMA bulk store), 20-21 P
// (mask A -> bf16 P), 22 TMA producer and issuer of MMA_A, 23 issuer of the
// other products and TMEM owner.  Every pipeline wait is bounded
// (gla_ptx.cuh).
//
// Strong gates: alpha has no lower bound, and once a channel decays by more
// than e^-64 over a chunk the factor e^{-b_i} could overflow.  The pass every
// call runs only detects such a chunk; the CTA then skips its final-state write
// and runs its slice a second time (exact_pass) in which strong channels take
// k e^{b_C - b_i} (already decayed to the chunk end, <= 1) and their
// intra-chunk scores are added on the P warps with exponents <= 0.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "gla_internal.h"
#include "gla_ptx.cuh"

// Optional per-role timestamps of CTA 0 (compiled in only with -DGLA_TRACE).
#ifdef GLA_TRACE
__device__ unsigned long long* g_gla_trace;
#define GLA_TRACE_POINT(ev, c)                                                           \
    do {                                                                                 \
        if (blockIdx.x == 0 && g_gla_trace && (c) < 512) g_gla_trace[(ev) * 512 + (c)] = \
            gla::globaltimer();                                                          \
    } while (0)
#else
#define GLA_TRACE_POINT(ev, c) \
    do {                       \
    } while (0)
#endif

namespace gla {
namespace {

constexpr int C = 64;  // chunk length (tokens)
constexpr int NS_MAX = 4;  // q/k stages at most (hold Qh/Kh until the chunk's MMAs finish)
constexpr int NV_MAX = 4;  // V stages at most
constexpr int NL = 2;  // log-alpha stages
constexpr int kWarps = 24;
constexpr int kThreads = kWarps * 32;
constexpr int W_STATE0 = 8, W_OUT0 = 16, W_P0 = 20, W_TMA = 22, W_MMA = 23;
constexpr int kGateThreads = 256;

// A key channel whose gate decays by more than e^-64 over one chunk is "strong"
// for that chunk: the factor k e^{-b_i} could overflow, so such channels take
// k e^{b_C - b_i} (the state update then adds their dS after the decay) and
// their intra-chunk scores are added on the P warps with exponents <= 0 (see
// gate_factors_strong, strong_scores).  The test is made on e^{b_C} exactly as
// the gate writes it, so every role agrees.
constexpr float kStrongGamma = 1.6038109e-28f;  // e^-64
constexpr float kStrongLog = -64.f;
constexpr int kRing = 8;  // chunks whose strong-channel masks are kept (ring slots)

// tensor-memory column map (512 columns allocated)
constexpr uint32_t TM_S = 0;     // S^T fp32, dk columns (128-column tile)
constexpr uint32_t TM_DS = 128;  // dS^T fp32, dk columns
constexpr uint32_t TM_SB = 256;  // bf16 copy of S^T for the next O_i, dk/2 columns (128-column tile)
// With the 64-column tile (M = 64) S^T is held in the state warps'
// registers instead, and the map is: two dS^T buffers at 0..127 and
// 128..255 (dS(c) in buffer c & 1, released by the state warps once read),
// O^T 2 x 64 at 256..383, the bf16 copy of the state at 384..447 (key
// channels 2x, 2x + 1 in column x), A at 448..511.  The copy of the state
// after chunk c, read by O_i(c + 1), is written once O_i(c) has read the
// previous one: only the copy write waits on a product, never the fp32 state
// update, and a dS buffer waits only on the state warps' read.
constexpr uint32_t TM_CP64 = 384;  // 64-column tile: bf16 copy of S^T, 64 columns
constexpr uint32_t TM_O = 320;   // 2 x O^T fp32, 64 columns each
constexpr uint32_t TM_A = 448;   // A fp32, 64 columns
constexpr uint32_t TM_COLS = 512;

template <int DVT>
struct VRing {
    static constexpr int N = DVT == 64 ? 3 : 2;
};

enum {
    B_QK_FULL = 0,
    B_QK_GATED = B_QK_FULL + NS_MAX,
    B_QK_EMPTY = B_QK_GATED + NS_MAX,
    B_LA_FULL = B_QK_EMPTY + NS_MAX,
    B_LA_EMPTY = B_LA_FULL + NL,
    B_V_FULL = B_LA_EMPTY + NL,
    B_V_EMPTY = B_V_FULL + NV_MAX,
    B_A_FULL = B_V_EMPTY + NV_MAX,
    B_A_EMPTY,
    B_P_FULL,    // 2
    B_P_EMPTY = B_P_FULL + 2,  // 2
    B_DS_FULL = B_P_EMPTY + 2,    // 2 (one per dS buffer; the 128-column tile uses one)
    B_DS_EMPTY = B_DS_FULL + 2,   // 2
    B_S_READY = B_DS_EMPTY + 2,   // 2
    B_SB_EMPTY = B_S_READY + 2,  // 2
    B_O_FULL = B_SB_EMPTY + 2,   // 2
    B_O_EMPTY = B_O_FULL + 2,  // 2
    B_DRAIN = B_O_EMPTY + 2,
    B_STALL,  // completed by nothing: the test-only stall waits on it
    // 64-column tile only (last, so that the 128-column tile's layout does not hold them):
    // e^{b_C} (and the strong masks) of chunk c written to slot c % kRing
    B_G_READY,
    B_COUNT = B_G_READY + kRing
};

// SCALAR: one log alpha per token (shared by all channels): its tile is 256
// bytes instead of DK * 256, and the shared memory it frees buys a fourth q/k
// stage and a deeper V ring.
template <int DK, int DVT, bool SCALAR = false>
struct Layout {
    static constexpr int NS = SCALAR ? 4 : 3;
    static constexpr int NV = SCALAR ? (DVT == 64 ? 4 : 3) : VRing<DVT>::N;
    static constexpr int QB = DK * C * 2;        // one bf16 [64][DK] tile (DK/64 swizzle atoms)
    static constexpr int STAGE_QK = 2 * QB;
    static constexpr int LAB = SCALAR ? C * 4 : DK * C * 4;  // fp32 [64][DK], or [64] with SCALAR
    static constexpr int LA_REGION = (NL * LAB + 1023) / 1024 * 1024;  // the V tiles stay 1024-aligned
    static constexpr int VB = DVT * C * 2;       // bf16 [64][DVT] as DVT/64 atoms of 64 columns
    static constexpr int PB = C * C * 2;         // bf16 [64][64]
    static constexpr int OSB = C * DVT * 2;      // output staging, DVT/64 blocks of [64][64] bf16
    static constexpr int QUADS = DK / 4;
    static constexpr int SEG = kGateThreads / QUADS;  // token segments in the gate mapping
    static constexpr int TPS = C / SEG;               // tokens per segment
    static constexpr int off_qk = 0;
    static constexpr int off_la = off_qk + NS * STAGE_QK;
    static constexpr int off_v = off_la + LA_REGION;
    // a second P buffer where it fits: P(c+1) need not wait for O_a(c)
    // e^{b_C} slots: a ring of its own with the 64-column tile, one per q/k stage with the
    // 128-column tile (whose state update finishes before the stage is released)
    static constexpr int NG = DVT == 64 ? kRing : NS;
    static constexpr int NBAR = DVT == 64 ? B_COUNT : B_G_READY;
    static constexpr int NP = NS * STAGE_QK + LA_REGION + NV * VB + 2 * PB + OSB + NG * DK * 4 + 2 * SEG * DK * 4 +
                                      NBAR * 8 + 16 + kRing * 20 + 1008 <= 232448
                                  ? 2
                                  : 1;
    static constexpr int off_p = off_v + NV * VB;
    static constexpr int off_ost = off_p + NP * PB;
    static constexpr int off_gamma = off_ost + OSB;
    static constexpr int off_segtot = off_gamma + NG * DK * 4;  // e^{b_C} of chunk c in slot c % NG
    static constexpr int off_bar = off_segtot + 2 * SEG * DK * 4;
    static constexpr int off_misc = off_bar + NBAR * 8;
    // ring of per-chunk strong-channel masks: {sequence, 4 x 32-bit masks} per slot
    static constexpr int off_ring = off_misc + 16;
    static constexpr int total = off_ring + kRing * 20;  // misc: TMEM base address, abort flag, O_i count
    static constexpr int alloc = total + 1008;  // round-up to 1024 from a >= 16-byte aligned base
    static_assert(alloc <= 232448, "shared memory budget");
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_la, tm_v, tm_out;
    const uint16_t* q_raw;  // the same inputs as plain pointers (strong-channel scores)
    const uint16_t* k_raw;
    const float* la_raw;
    const float* init_state;
    const float* init_z;
    void* out;
    float* final_state;
    float* final_z;
    unsigned* err;
    unsigned long long wait_ns;  // limit of the pipeline waits (the drain waits keep kWaitLimitNs)
    int test_stall;              // gate role first waits on B_STALL (error-path tests)
    int L, dv, nchunks, ntile;
    unsigned flags;
    int out_f32;
};

// TMEM lane <-> value column within the CTA's DVT slice.  M = 128: lane j is
// column j.  M = 64: column 16q + r sits in lane 32q + r (r < 16).
template <int DVT>
__device__ __forceinline__ int lane_to_col(int warp_quarter, int lane) {
    if (DVT == 128) return warp_quarter * 32 + lane;
    return lane < 16 ? warp_quarter * 16 + lane : -1;
}

// Packed fp32 pair add and multiply (one instruction each, IEEE round-to-nearest,
// bit-identical to the scalar forms).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
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

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Gate factor phase of one gate thread: TPS tokens (its segment) x 4 key
// channels.  `off` holds the prefix of the earlier segments (b before the
// segment) in natural log units; the running value b_t is kept in log2 units so
// that each factor is a single ex2:  Qh = q * 2^{b_t log2 e},  Kh = k * 2^{-b_t log2 e}.
// The feature map and the gate are compile-time branches so that the token
// loop stays one basic block the scheduler can interleave.
// With SCALAR (one log alpha per token) all four channels share one running
// value, so a token costs one pair of ex2 instead of four.
template <int DK, int TPS, int G, bool GATE, bool ELU, bool SCALAR>
__device__ __forceinline__ void gate_factors(uint8_t* qt, uint8_t* kt, const float* la, int seg, int col, int nval,
                                             const float (&off)[4]) {
    constexpr float kLog2e = 1.4426950408889634f;
    const float2 l2e = make_float2(kLog2e, kLog2e);
    float2 run01 = make_float2(off[0] * kLog2e, off[1] * kLog2e), run23 = make_float2(off[2] * kLog2e, off[3] * kLog2e);
    float run_s = off[0] * kLog2e;
#pragma unroll 1
    for (int i0 = 0; i0 < TPS; i0 += G) {
        uint2 qr[G], kr[G];
        float4 lx[G];
#pragma unroll
        for (int u = 0; u < G; u++) {
            const int t = seg * TPS + i0 + u;
            const uint32_t o = sw128_offset(t, col);
            qr[u] = *reinterpret_cast<const uint2*>(qt + o);
            kr[u] = *reinterpret_cast<const uint2*>(kt + o);
            if (GATE) lx[u] = SCALAR ? make_float4(la[t], 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(la + t * DK);
        }
        if constexpr (GATE && !ELU) {
            // products as packed fp32 pairs (each rounded once to bf16, as the scalar form)
#pragma unroll
            for (int u = 0; u < G; u++) {
                float2 f_q01, f_q23, f_k01, f_k23;
                if (SCALAR) {
                    run_s = fmaf(lx[u].x, kLog2e, run_s);
                    const float fq = ex2_approx(run_s), fk = ex2_approx(-run_s);
                    f_q01 = f_q23 = make_float2(fq, fq);
                    f_k01 = f_k23 = make_float2(fk, fk);
                } else {
                    run01 = fma2(make_float2(lx[u].x, lx[u].y), l2e, run01);
                    run23 = fma2(make_float2(lx[u].z, lx[u].w), l2e, run23);
                    f_q01 = make_float2(ex2_approx(run01.x), ex2_approx(run01.y));
                    f_q23 = make_float2(ex2_approx(run23.x), ex2_approx(run23.y));
                    f_k01 = make_float2(ex2_approx(-run01.x), ex2_approx(-run01.y));
                    f_k23 = make_float2(ex2_approx(-run23.x), ex2_approx(-run23.y));
                }
                const float2 q01 = unpack_bf16x2(qr[u].x), q23 = unpack_bf16x2(qr[u].y);
                const float2 k01 = unpack_bf16x2(kr[u].x), k23 = unpack_bf16x2(kr[u].y);
                const float2 a = mul2(q01, f_q01), b = mul2(q23, f_q23), c = mul2(k01, f_k01), d = mul2(k23, f_k23);
                qr[u] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(b.x, b.y));
                kr[u] = make_uint2(pack_bf16x2(c.x, c.y), pack_bf16x2(d.x, d.y));
            }
        } else {
#pragma unroll
            for (int u = 0; u < G; u++) {
                float2 q01 = unpack_bf16x2(qr[u].x), q23 = unpack_bf16x2(qr[u].y);
                float2 k01 = unpack_bf16x2(kr[u].x), k23 = unpack_bf16x2(kr[u].y);
                if (ELU) {
                    q01 = make_float2(elu1(q01.x), elu1(q01.y));
                    q23 = make_float2(elu1(q23.x), elu1(q23.y));
                    k01 = make_float2(elu1(k01.x), elu1(k01.y));
                    k23 = make_float2(elu1(k23.x), elu1(k23.y));
                }
                float2 fq01 = make_float2(1.f, 1.f), fq23 = fq01, fk01 = fq01, fk23 = fq01;
                if (GATE && SCALAR) {  // run = b_t log2 e <= 0, the same for every channel
                    run_s = fmaf(lx[u].x, kLog2e, run_s);
                    const float fq = ex2_approx(run_s), fk = ex2_approx(-run_s);
                    fq01 = fq23 = make_float2(fq, fq);
                    fk01 = fk23 = make_float2(fk, fk);
                } else if (GATE) {  // run = b_t log2 e <= 0
                    run01 = fma2(make_float2(lx[u].x, lx[u].y), l2e, run01);
                    run23 = fma2(make_float2(lx[u].z, lx[u].w), l2e, run23);
                    fq01 = make_float2(ex2_approx(run01.x), ex2_approx(run01.y));
                    fq23 = make_float2(ex2_approx(run23.x), ex2_approx(run23.y));
                    fk01 = make_float2(ex2_approx(-run01.x), ex2_approx(-run01.y));
                    fk23 = make_float2(ex2_approx(-run23.x), ex2_approx(-run23.y));
                }
                if (GATE) {
                    // the feature map's path keeps scalar products (packed pairs spill here)
                    q01 = make_float2(q01.x * fq01.x, q01.y * fq01.y);
                    q23 = make_float2(q23.x * fq23.x, q23.y * fq23.y);
                    k01 = make_float2(k01.x * fk01.x, k01.y * fk01.y);
                    k23 = make_float2(k23.x * fk23.x, k23.y * fk23.y);
                }
                qr[u] = make_uint2(pack_bf16x2(q01.x, q01.y), pack_bf16x2(q23.x, q23.y));
                kr[u] = make_uint2(pack_bf16x2(k01.x, k01.y), pack_bf16x2(k23.x, k23.y));
                // rows past the sequence end arrive zero-filled; only phi(0) = 1 needs masking
                if (ELU && seg * TPS + i0 + u >= nval) qr[u] = kr[u] = make_uint2(0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < G; u++) {
            const uint32_t o = sw128_offset(seg * TPS + i0 + u, col);
            *reinterpret_cast<uint2*>(qt + o) = qr[u];
            *reinterpret_cast<uint2*>(kt + o) = kr[u];
        }
    }
}

// The four log gates of this thread's channels at token t (one shared gate with SCALAR).
template <int DK, bool SCALAR>
__device__ __forceinline__ float4 load_la4(const float* la, int t) {
    if (SCALAR) {
        const float x = la[t];
        return make_float4(x, x, x, x);
    }
    return *reinterpret_cast<const float4*>(la + t * DK);
}

// Gate factors of a thread that owns at least one strong channel in this chunk
// (its gate decays by more than e^-64 over the chunk, so k e^{-b_t} could
// overflow).  q takes e^{b_t} on every channel; on strong channels k takes
// e^{b_C - b_t} (<= 1, already decayed to the chunk end), accumulated as a
// suffix sum from the chunk end so that it stays exact however large |b_C| is;
// the thread's other channels keep k e^{-b_t}.
//   pre: sum of log alpha over the segments before this thread's, suf: over the
//   segments after it, tot: over the whole chunk (b_C).
template <int DK, int TPS, bool ELU, bool SCALAR>
__device__ __noinline__ void gate_factors_strong(uint8_t* qt, uint8_t* kt, const float* la, int seg, int col,
                                                 int nval, float4 pre, float4 tot, float4 suf, unsigned strong4) {
    constexpr float kLog2e = 1.4426950408889634f;
    float rq[4] = {pre.x, pre.y, pre.z, pre.w};
    float rk[4] = {(strong4 & 1u) ? suf.x : suf.x - tot.x, (strong4 & 2u) ? suf.y : suf.y - tot.y,
                   (strong4 & 4u) ? suf.z : suf.z - tot.z, (strong4 & 8u) ? suf.w : suf.w - tot.w};
#pragma unroll 1
    for (int i = 0; i < TPS; i++) {  // q: forward running sum b_t
        const int t = seg * TPS + i;
        const float4 x = load_la4<DK, SCALAR>(la, t);
        rq[0] += x.x;
        rq[1] += x.y;
        rq[2] += x.z;
        rq[3] += x.w;
        const uint32_t o = sw128_offset(t, col);
        const uint2 qr = *reinterpret_cast<const uint2*>(qt + o);
        float2 q01 = unpack_bf16x2(qr.x), q23 = unpack_bf16x2(qr.y);
        if (ELU) {
            q01 = make_float2(elu1(q01.x), elu1(q01.y));
            q23 = make_float2(elu1(q23.x), elu1(q23.y));
        }
        q01.x *= ex2_approx(rq[0] * kLog2e);
        q01.y *= ex2_approx(rq[1] * kLog2e);
        q23.x *= ex2_approx(rq[2] * kLog2e);
        q23.y *= ex2_approx(rq[3] * kLog2e);
        uint2 w = make_uint2(pack_bf16x2(q01.x, q01.y), pack_bf16x2(q23.x, q23.y));
        if (ELU && t >= nval) w = make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(qt + o) = w;
    }
#pragma unroll 1
    for (int i = TPS - 1; i >= 0; i--) {  // k: suffix sum b_C - b_t (- b_C off the strong channels)
        const int t = seg * TPS + i;
        const uint32_t o = sw128_offset(t, col);
        const uint2 kr = *reinterpret_cast<const uint2*>(kt + o);
        float2 k01 = unpack_bf16x2(kr.x), k23 = unpack_bf16x2(kr.y);
        if (ELU) {
            k01 = make_float2(elu1(k01.x), elu1(k01.y));
            k23 = make_float2(elu1(k23.x), elu1(k23.y));
        }
        k01.x *= ex2_approx(rk[0] * kLog2e);
        k01.y *= ex2_approx(rk[1] * kLog2e);
        k23.x *= ex2_approx(rk[2] * kLog2e);
        k23.y *= ex2_approx(rk[3] * kLog2e);
        uint2 w = make_uint2(pack_bf16x2(k01.x, k01.y), pack_bf16x2(k23.x, k23.y));
        if (ELU && t >= nval) w = make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(kt + o) = w;
        const float4 x = load_la4<DK, SCALAR>(la, t);
        rk[0] += x.x;
        rk[1] += x.y;
        rk[2] += x.z;
        rk[3] += x.w;
    }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Intra-chunk scores of the strong channels of a chunk, added in place to row t
// of the A tile in tensor memory (both 32-column halves):
//   A[t][i] += sum_{d strong} q_td k_id e^{b_td - b_id}   for i <= t.
// (The tensor-core product carries these channels with the factors e^{b_t} and
// e^{b_C - b_i}, whose product is below e^-64 |q_td k_id|: nothing.)  The
// exponent is a running sum of log alpha walked from i = t downwards, so it is
// <= 0 and exact for any gate; the walk stops once it is below -88.  Raw q, k
// and log alpha are read from global memory (the chunk was loaded a moment ago,
// so they come from L2).  Called by whole warps (the tensor-memory accesses are
// warp-collective) and only for chunks with a strong channel.
template <int DK, bool SCALAR>
__device__ __noinline__ void strong_scores(uint32_t taddr, int t, int nval, uint4 mask4, const uint16_t* qc,
                                           const uint16_t* kc, const float* lac, bool elu) {
    const uint32_t mask[4] = {mask4.x, mask4.y, mask4.z, mask4.w};
    auto lag = [&](int j, int d) { return SCALAR ? lac[j] : lac[(long)j * DK + d]; };
#pragma unroll 1
    for (int h = 0; h < 2; h++) {
        uint32_t r[32];
        tmem_ld32(taddr + h * 32, r);
        tmem_wait_ld();
        const int top = min(t, 32 * h + 31);
        // rows past the sequence end are never stored; columns above the diagonal are masked
        if (t < nval && top >= 32 * h) {
#pragma unroll 1
            for (int e4 = 0; e4 < 4; e4++) {
                uint32_t m = mask[e4];  // bit `quad` set: channel 4 quad + e4 is strong
#pragma unroll 1
                while (m) {
                    const int quad = __ffs(m) - 1;
                    m &= m - 1;
                    const int d = 4 * quad + e4;
                    float qd = bf16_bits_to_float(qc[(long)t * DK + d]);
                    if (elu) qd = elu1(qd);
                    float s = 0.f;  // b_t - b_i for i = top
#pragma unroll 1
                    for (int j = t; j > top && s >= -88.f; j--) s += lag(j, d);
                    if (s < -88.f) continue;
#pragma unroll
                    for (int e = 31; e >= 0; e--) {
                        const int i = 32 * h + e;
                        if (i <= top) {
                            float kd = bf16_bits_to_float(kc[(long)i * DK + d]);
                            if (elu) kd = elu1(kd);
                            r[e] = __float_as_uint(
                                fmaf(qd * kd, ex2_approx(s * 1.4426950408889634f), __uint_as_float(r[e])));
                            s += lag(i, d);
                            if (s < -88.f) break;
                        }
                    }
                }
            }
        }
        __syncwarp();
        tmem_st32(taddr + h * 32, r);
        tmem_wait_st();
    }
}

// Wait (bounded) until the gate has published the strong-channel masks of chunk c.
__device__ __forceinline__ bool ring_wait(const volatile uint32_t* slot, uint32_t c, volatile int* abort_flag,
                                          unsigned* err_word, unsigned long long limit_ns) {
    if (slot[0] == c) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (slot[0] == c) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                if (err_word) record_timeout_code(err_word, 0x10000000u | ((c & 0xffffu) << 1));
                return false;
            }
        }
    }
}

// One pass of a CTA over its (batch*head, value slice).
// SAFE = false: the pass every call makes.  A chunk whose gate decays by more
// than e^-64 on some channel is not computed exactly by the factorisation
// (k e^{-b_t} could overflow); such a chunk only raises a flag, the pass then
// skips the final-state write and returns true (its outputs are rewritten).
// SAFE = true: the pass that follows in the same CTA when the first returned
// true; it recomputes the slice with strong channels handled exactly
// (gate_factors_strong, strong_scores).  Tensor memory is allocated once by
// the kernel for both passes.
template <int DK, int DVT, bool GATE, bool SCALAR, bool SAFE>
__device__ __forceinline__ bool prefill_pass(const TcParams& p, uint8_t* smem_raw) {
    using Ly = Layout<DK, DVT, SCALAR>;
    constexpr int NS = Ly::NS;
    constexpr int NV = Ly::NV;
    // 1024-byte aligned base for the swizzled tiles.  The offset is added to the
    // shared array itself so that every access below stays in the shared
    // address space (an integer round trip would turn them into generic ones).
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::off_bar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Ly::off_misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Ly::off_misc + 4);
    // number of O_i products issued so far (written by the MMA thread, read by the A issuer)
    volatile int* oi_issued = reinterpret_cast<volatile int*>(sm + Ly::off_misc + 8);
    // fast pass: set once some chunk of this slice has a strong channel
    volatile int* strong_flag = reinterpret_cast<volatile int*>(sm + Ly::off_misc + 12);
    float* gamma = reinterpret_cast<float*>(sm + Ly::off_gamma);
    // slot c % kRing: {chunk index, strong-channel masks m[4]}; bit `quad` of m[e] is channel 4 quad + e
    uint32_t* ring = reinterpret_cast<uint32_t*>(sm + Ly::off_ring);
    float* segtot = reinterpret_cast<float*>(sm + Ly::off_segtot);
    // normaliser denominators: only with GLA_FLAG_NORMALIZE (dv == 64 on a 128-column
    // tile), when the second 64-column block of the output staging is unused
    float* den = reinterpret_cast<float*>(sm + Ly::off_ost + 8192);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // A(c) comes from the TMA producer thread, the other three products from the MMA thread
    constexpr uint32_t kTmO = DVT == 64 ? 256u : TM_O;  // the two O^T buffers
    const int tile = blockIdx.x % p.ntile;
    const int bh = blockIdx.x / p.ntile;
    const int j0 = tile * DVT;
    const int L = p.L, dv = p.dv, N = p.nchunks;
    const bool norm = p.flags & GLA_FLAG_NORMALIZE;
    const bool elu = p.flags & GLA_FLAG_FEATURE_ELU1;
    // value columns holding real data; with the normaliser (dv == 64, DVT == 128) column 64 holds z
    const int jvalid = min(DVT, dv - j0);
    const int nvb = jvalid / 64;  // TMA-loaded 64-column blocks of V

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        if (SAFE)  // the first pass's barriers are re-initialised
            for (int i = 0; i < B_COUNT; i++) mbar_inval(bar(i));
        for (int i = 0; i < NS; i++) {
            mbar_init(bar(B_QK_FULL + i), 1);
            mbar_init(bar(B_QK_GATED + i), 8);
            mbar_init(bar(B_QK_EMPTY + i), 2);  // released by the issuers of A (TMA thread) and of dS, O_i
        }
        for (int i = 0; i < NL; i++) {
            mbar_init(bar(B_LA_FULL + i), 1);
            mbar_init(bar(B_LA_EMPTY + i), 8);
        }
        for (int i = 0; i < NV; i++) {
            mbar_init(bar(B_V_FULL + i), 1);
            mbar_init(bar(B_V_EMPTY + i), 1);
        }
        mbar_init(bar(B_A_FULL), 1);
        mbar_init(bar(B_A_EMPTY), 2);
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_P_FULL + i), 2);
            mbar_init(bar(B_P_EMPTY + i), 1);
            mbar_init(bar(B_SB_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_DS_FULL + i), 1);
            mbar_init(bar(B_DS_EMPTY + i), 8);  // released by the state warps once they have read dS
        }
        mbar_init(bar(B_S_READY), 8);
        mbar_init(bar(B_S_READY + 1), 8);
        mbar_init(bar(B_O_FULL), 1);
        mbar_init(bar(B_O_FULL + 1), 1);
        mbar_init(bar(B_O_EMPTY), 4);
        mbar_init(bar(B_O_EMPTY + 1), 4);
        if (DVT == 64)
            for (int i = 0; i < kRing; i++) mbar_init(bar(B_G_READY + i), 8);
        mbar_init(bar(B_DRAIN), 2);
        mbar_init(bar(B_STALL), 1);
        *abort_flag = 0;
        *oi_issued = 0;
        *strong_flag = 0;
        for (int i = 0; i < kRing; i++) ring[i * 5] = 0xffffffffu;
        mbar_fence_init();
    }
    if (!SAFE && warp == W_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    // V columns the TMA never writes (dv == 64 on a 128-column tile): zero,
    // plus the all-ones normaliser column
    if (DVT == 128 && nvb < 2) {
        for (int idx = threadIdx.x; idx < NV * C * 64; idx += kThreads) {
            const int st = idx / (C * 64), rem = idx % (C * 64);
            const int row = rem / 64, col = rem % 64;
            const float x = (norm && col == 0) ? 1.f : 0.f;
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(sm + Ly::off_v + st * Ly::VB + 8192 +
                                                                  sw128_offset(row, col));
            *dst = __float2bfloat16_rn(x);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_field = static_cast<uint32_t>((warp & 3) * 32) << 16;

    int pl_n = 0, pq_n = 0, pv_n = 0;  // producer: chunks whose log-alpha / q,k / v loads were issued

    if (warp < W_STATE0) {
        // ============================================================ gate
        constexpr int QUADS = Ly::QUADS, SEG = Ly::SEG, TPS = Ly::TPS;
        constexpr int G = TPS < 2 ? TPS : 2;  // tokens per factor group (2: no register spills)
        const int gt = threadIdx.x;
        const int quad = gt % QUADS, seg = gt / QUADS;
        const int ch = 4 * quad;
        const int atom = ch >> 6, col = ch & 63;
        // error-path tests: a wait that nothing completes runs out and stops every role
        bool ok0 = true;
        if (p.test_stall) ok0 = mbar_wait(bar(B_STALL), 0, abort_flag, p.err, p.wait_ns);
        for (int c = 0; c < N; c++) {
            const int s = c % NS, l = c % NL;
            bool ok = ok0;
            if (GATE && ok) ok = mbar_wait(bar(B_LA_FULL + l), (c / NL) & 1, abort_flag, p.err, p.wait_ns);
            if (ok) ok = mbar_wait(bar(B_QK_FULL + s), (c / NS) & 1, abort_flag, p.err, p.wait_ns);
            if (threadIdx.x == 0) GLA_TRACE_POINT(0, c);
            // Phase 1: per-segment cumulative sums of log alpha, exchanged across the
            // gate warps to give each thread the prefix before its segment (off) and
            // the chunk total b_C (tot).  Phase 2 re-reads log alpha from shared
            // memory and re-accumulates, so no per-token sums are held in registers.
            float off[4] = {0.f, 0.f, 0.f, 0.f}, tot[4] = {0.f, 0.f, 0.f, 0.f}, pre[4] = {0.f, 0.f, 0.f, 0.f};
            unsigned strong4 = 0;  // strong channels among this thread's four
            // per-channel: this thread's 4 channels of row t at la + t*DK; SCALAR: row t at la[t]
            const float* la = reinterpret_cast<const float*>(sm + Ly::off_la + l * Ly::LAB) + (SCALAR ? 0 : ch);
            if (GATE) {
                float* st = segtot + (c & 1) * SEG * DK;
                if (ok) {
                    float2 r01 = make_float2(0.f, 0.f), r23 = r01;
#pragma unroll
                    for (int i = 0; i < TPS; i++) {
                        const float4 x = SCALAR ? make_float4(la[seg * TPS + i], la[seg * TPS + i], la[seg * TPS + i],
                                                              la[seg * TPS + i])
                                                : *reinterpret_cast<const float4*>(la + (seg * TPS + i) * DK);
                        r01 = add2(r01, make_float2(x.x, x.y));
                        r23 = add2(r23, make_float2(x.z, x.w));
                    }
                    *reinterpret_cast<float4*>(st + seg * DK + ch) = make_float4(r01.x, r01.y, r23.x, r23.y);
                }
                // the segment-total exchange doubles as the gate role's agreement to go on
                if (!bar_red_and(1, kGateThreads, ok)) break;
                {
                    // all segment totals in flight at once; the prefix takes those before this
                    // thread's segment (seg is the warp index: the test is warp-uniform)
                    float2 o01 = make_float2(0.f, 0.f), o23 = o01, t01 = o01, t23 = o01;
                    // the chunk total is needed by segment 0 only (e^{b_C}, the strong test),
                    // except in the exact pass, where every thread tests its own channels
                    const bool need_tot = SAFE || seg == 0;
#pragma unroll
                    for (int g = 0; g < SEG; g++) {
                        if (!(g < seg || need_tot)) continue;
                        const float4 u = *reinterpret_cast<const float4*>(st + g * DK + ch);
                        if (g < seg) {
                            o01 = add2(o01, make_float2(u.x, u.y));
                            o23 = add2(o23, make_float2(u.z, u.w));
                        } else {
                            t01 = add2(t01, make_float2(u.x, u.y));
                            t23 = add2(t23, make_float2(u.z, u.w));
                        }
                    }
                    t01 = add2(t01, o01);
                    t23 = add2(t23, o23);
                    off[0] = o01.x; off[1] = o01.y; off[2] = o23.x; off[3] = o23.y;
                    tot[0] = t01.x; tot[1] = t01.y; tot[2] = t23.x; tot[3] = t23.y;
                }
                if constexpr (SAFE) {
                    // e^{b_C} per channel: the state's decay; below e^-64 the channel is strong
                    const float4 gm4 = make_float4(__expf(tot[0]), __expf(tot[1]), __expf(tot[2]), __expf(tot[3]));
                    strong4 = (gm4.x < kStrongGamma ? 1u : 0u) | (gm4.y < kStrongGamma ? 2u : 0u) |
                              (gm4.z < kStrongGamma ? 4u : 0u) | (gm4.w < kStrongGamma ? 8u : 0u);
                    if (seg == 0) *reinterpret_cast<float4*>(gamma + (c % Ly::NG) * DK + ch) = gm4;
                    if (warp == 0) {  // every segment-0 thread (one per channel quad) is in warp 0
                        uint32_t m[4];
    #pragma unroll
                        for (int e = 0; e < 4; e++) m[e] = __ballot_sync(0xffffffffu, seg == 0 && ((strong4 >> e) & 1u));
                        if (lane == 0) {
                            uint32_t* slot = ring + (c % kRing) * 5;
    #pragma unroll
                            for (int e = 0; e < 4; e++) slot[1 + e] = m[e];
                            __threadfence_block();
                            *reinterpret_cast<volatile uint32_t*>(slot) = static_cast<uint32_t>(c);
                        }
                    }
                } else {
                    if (seg == 0)
                        *reinterpret_cast<float4*>(gamma + (c % Ly::NG) * DK + ch) =
                            make_float4(__expf(tot[0]), __expf(tot[1]), __expf(tot[2]), __expf(tot[3]));
                    if (seg == 0 && fminf(fminf(tot[0], tot[1]), fminf(tot[2], tot[3])) < kStrongLog) *strong_flag = 1;
                }
#pragma unroll
                for (int e = 0; e < 4; e++) pre[e] = off[e];  // the running value is b_t
            } else {
                if (!bar_red_and(1, kGateThreads, ok)) break;
            }
            if (threadIdx.x == 0) GLA_TRACE_POINT(2, c);
            // 64-column tile: e^{b_C} of chunk c is in its slot, the state update may start.
            // (The slots outlive the q/k stage: the gate is at most NS + 1 chunks ahead of
            // the last finished state update, since a stage is reloaded only after its O_i,
            // which read the state after the chunk before.)
            if (GATE && DVT == 64) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_G_READY + c % kRing));
            }
            const int nval = min(C, L - c * C);
            // Rows past the sequence end arrive zero-filled (q, k and log alpha), so they
            // add nothing to A, dS or O; only the feature map (phi(0) = 1) needs them masked.
            if (GATE || elu) {
                uint8_t* qt = sm + Ly::off_qk + s * Ly::STAGE_QK + atom * 8192;
                uint8_t* kt = qt + Ly::QB;
                if (SAFE && GATE && strong4) {  // only the exact pass sets strong4
                    // suffix of the chunk after this thread's segment (still in segtot)
                    const float* st = segtot + (c & 1) * SEG * DK;
                    float4 suf = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int g = seg + 1; g < SEG; g++) {
                        const float4 u = *reinterpret_cast<const float4*>(st + g * DK + ch);
                        suf.x += u.x;
                        suf.y += u.y;
                        suf.z += u.z;
                        suf.w += u.w;
                    }
                    const float4 pre4 = make_float4(pre[0], pre[1], pre[2], pre[3]);
                    const float4 tot4 = make_float4(tot[0], tot[1], tot[2], tot[3]);
                    if (elu)
                        gate_factors_strong<DK, TPS, true, SCALAR>(qt, kt, la, seg, col, nval, pre4, tot4, suf,
                                                                   SAFE ? strong4 : 0u);
                    else
                        gate_factors_strong<DK, TPS, false, SCALAR>(qt, kt, la, seg, col, nval, pre4, tot4, suf,
                                                                    SAFE ? strong4 : 0u);
                } else if (elu) {
                    gate_factors<DK, TPS, G, GATE, true, SCALAR>(qt, kt, la, seg, col, nval, off);
                } else {
                    gate_factors<DK, TPS, G, GATE, false, SCALAR>(qt, kt, la, seg, col, nval, off);
                }
            }
            if (GATE) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_LA_EMPTY + l));
            }
            if (threadIdx.x == 0) GLA_TRACE_POINT(14, c);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QK_GATED + s));
            if (threadIdx.x == 0) GLA_TRACE_POINT(3, c);
        }
    } else if (warp < W_OUT0) {
        // ============================================================ state
        constexpr int COLS = DK / 2;  // key channels per warp (two warps per lane quarter)
        const int half = (warp - W_STATE0) >> 2;
        const int cbase = half * COLS;
        if constexpr (DVT == 64) {
            // S^T in registers.  M = 64 rows sit in lanes 0-15 of each quarter; with the
            // 16x32bx2 TMEM shape threads 0-15 and 16-31 take the same 16 rows at two
            // column offsets, so the whole warp works: thread (r, hi) owns row r and the
            // key channels cbase + 32 g + 16 hi + [0, 16).
            constexpr int NG = COLS / 32;
            const int hi = lane >> 4;
            const int jl = lane_to_col<DVT>(warp & 3, lane & 15);
            const int j = j0 + jl;
            const bool jv = jl < jvalid;
            float S[NG * 16];
            {
                const float* s0 = (p.init_state && jv) ? p.init_state + (long)bh * DK * dv + j : nullptr;
#pragma unroll
                for (int g = 0; g < NG; g++)
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        S[g * 16 + i] = s0 ? s0[(long)(cbase + g * 32 + hi * 16 + i) * dv] : 0.f;
            }
            // bf16 copy of the state for O_i: group g (8 key channels c0 + [0, 8) of this
            // half-warp, and c0 + 16 + [0, 8) for threads 16-31) goes to column c0 / 2
            const uint32_t tCP = tmem + lane_field + TM_CP64;
            auto write_copy = [&]() {
#pragma unroll
                for (int g = 0; g < NG * 2; g++) {
                    const int c0 = cbase + (g >> 1) * 32 + (g & 1) * 8;
                    const float* sv = S + g * 8;
                    uint32_t pk[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) pk[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
                    tmem_st16x2_x4<8>(tCP + c0 / 2, pk);
                }
            };
            write_copy();  // the initial state's, for O_i(0)
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_READY));
            bool ok = true;
            for (int c = 0; c < N; c++) {
                const int s = c % NS;
                ok = mbar_wait_warp(bar(B_DS_FULL + (c & 1)), (c >> 1) & 1, abort_flag, p.err, p.wait_ns);
                if (warp == W_STATE0 && lane == 0) GLA_TRACE_POINT(16, c);
                if (ok && GATE)
                    ok = mbar_wait_warp(bar(B_G_READY + c % kRing), (c / kRing) & 1, abort_flag, p.err, p.wait_ns);
                if (warp == W_STATE0 && lane == 0) GLA_TRACE_POINT(17, c);
                if (!ok) break;
                tc_fence_after();
                if (warp == W_STATE0 && lane == 0) GLA_TRACE_POINT(4, c);
                // dS(c): this half's key channels [cbase, cbase + COLS) occupy columns
                // [cbase, cbase + COLS) of buffer c & 1
                const uint32_t tB = tmem + lane_field + (uint32_t)(c & 1) * 128u;
                // S <- e^{b_C} (S + dS): dS carries k e^{-b_i}.  A chunk with a strong channel:
                // that channel's dS carries k e^{b_C - b_i} (already decayed), so S <- e^{b_C} S + dS
                const uint32_t* slot = ring + (c % kRing) * 5;
                const bool sgc = SAFE && GATE && ((slot[1] | slot[2] | slot[3] | slot[4]) != 0u);
                auto update = [&](auto strong_tag) {
                    constexpr bool ST = decltype(strong_tag)::value;
#pragma unroll
                    for (int gp = 0; gp < NG * 2; gp += 2) {
                        // two groups of 8 key channels per half-warp (c0 + [0, 8) for threads 0-15,
                        // c0 + 16 + [0, 8) for threads 16-31; S index g/2 * 16 + (g&1) * 8 + i)
                        uint32_t d[2][8];
#pragma unroll
                        for (int u = 0; u < 2; u++)
                            tmem_ld16x2_x8<16>(tB + cbase + ((gp + u) >> 1) * 32 + ((gp + u) & 1) * 8, d[u]);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            const int g = gp + u;
                            const int c0 = cbase + (g >> 1) * 32 + (g & 1) * 8;
                            const float* gm = gamma + (c % Ly::NG) * DK + c0 + hi * 16;
#pragma unroll
                            for (int i = 0; i < 8; i += 4) {
                                float4 gv = make_float4(1.f, 1.f, 1.f, 1.f);
                                if (GATE) gv = *reinterpret_cast<const float4*>(gm + i);
                                float* sv = S + g * 8 + i;
                                const float d0 = __uint_as_float(d[u][i]), d1 = __uint_as_float(d[u][i + 1]),
                                            d2 = __uint_as_float(d[u][i + 2]), d3 = __uint_as_float(d[u][i + 3]);
                                if (ST) {
                                    sv[0] = gv.x < kStrongGamma ? fmaf(sv[0], gv.x, d0) : (sv[0] + d0) * gv.x;
                                    sv[1] = gv.y < kStrongGamma ? fmaf(sv[1], gv.y, d1) : (sv[1] + d1) * gv.y;
                                    sv[2] = gv.z < kStrongGamma ? fmaf(sv[2], gv.z, d2) : (sv[2] + d2) * gv.z;
                                    sv[3] = gv.w < kStrongGamma ? fmaf(sv[3], gv.w, d3) : (sv[3] + d3) * gv.w;
                                } else {
                                    const float2 a01 = mul2(add2(make_float2(sv[0], sv[1]), make_float2(d0, d1)),
                                                            make_float2(gv.x, gv.y));
                                    const float2 a23 = mul2(add2(make_float2(sv[2], sv[3]), make_float2(d2, d3)),
                                                            make_float2(gv.z, gv.w));
                                    sv[0] = a01.x;
                                    sv[1] = a01.y;
                                    sv[2] = a23.x;
                                    sv[3] = a23.y;
                                }
                            }
                        }
                    }
                };
                if (sgc)
                    update(std::true_type{});
                else
                    update(std::false_type{});
                // dS(c) has been read: its buffer takes dS(c + 2)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_DS_EMPTY + (c & 1)));
                // the copy of the state after chunk c, once O_i(c) has read the previous one
                if (!mbar_wait_warp(bar(B_SB_EMPTY), c & 1, abort_flag, p.err, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                write_copy();
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S_READY + ((c + 1) & 1)));
                if (warp == W_STATE0 && lane == 0) GLA_TRACE_POINT(5, c);
            }
            // a marked slice leaves its final state to the exact pass (init_state may alias it)
            if (ok && p.final_state && jv && !(GATE && !SAFE && *strong_flag)) {
                float* fs = p.final_state + (long)bh * DK * dv + j;
#pragma unroll
                for (int g = 0; g < NG; g++)
#pragma unroll
                    for (int i = 0; i < 16; i++) fs[(long)(cbase + g * 32 + hi * 16 + i) * dv] = S[g * 16 + i];
            }
        } else {
            const int jl = lane_to_col<DVT>(warp & 3, lane);  // column in the slice
            const int j = j0 + jl;
            const uint32_t tS = tmem + lane_field + TM_S;
            const uint32_t tD = tmem + lane_field + TM_DS;
            {
                const float* s0 =
                    (p.init_state && jl < jvalid) ? p.init_state + (long)bh * DK * dv + j : nullptr;
                const bool zl = norm && jl == 64;
                for (int g = 0; g < COLS / 16; g++) {
                    uint32_t r[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int d = cbase + g * 16 + i;
                        float x = 0.f;
                        if (s0)
                            x = s0[(long)d * dv];
                        else if (zl && p.init_z)
                            x = p.init_z[(long)bh * DK + d];
                        r[i] = __float_as_uint(x);
                    }
                    tmem_st16(tS + cbase + g * 16, r);
                    // the initial state's bf16 copy feeds O_i(0)
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        pk[i / 2] = pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                    tmem_st8(tmem + lane_field + TM_SB + (cbase + g * 16) / 2, pk);
                }
                tmem_wait_st();
                // first phase of the dS buffer's release; the copy for O_i(0) is ready
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_DS_EMPTY));
                    mbar_arrive(bar(B_S_READY));
                }
            }
            bool ok = true;
            for (int c = 0; c < N; c++) {
                const int s = c % NS;
                ok = mbar_wait_warp(bar(B_DS_FULL), c & 1, abort_flag, p.err, p.wait_ns);
                if (ok && GATE)
                    ok = mbar_wait_warp(bar(B_QK_GATED + s), (c / NS) & 1, abort_flag, p.err, p.wait_ns);
                // the single bf16 copy (of the state before this chunk) is free once O_i(c) has
                // completed; it then takes the updated state for O_i(c + 1)
                if (ok) ok = mbar_wait_warp(bar(B_SB_EMPTY), c & 1, abort_flag, p.err, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tSB = tmem + lane_field + TM_SB;
                // S <- e^{b_C} (S + dS) (dS carries k e^{-b_i}); a strong channel's dS carries
                // k e^{b_C - b_i}: S <- e^{b_C} S + dS
                const uint32_t* slot = ring + (c % kRing) * 5;
                const bool sgc = SAFE && GATE && ((slot[1] | slot[2] | slot[3] | slot[4]) != 0u);
#pragma unroll 1
                for (int g = 0; g < COLS / 16; g++) {
                    const int c0 = cbase + g * 16;
                    uint32_t rs[16], rd[16];
                    tmem_ld16(tS + c0, rs);
                    tmem_ld16(tD + c0, rd);
                    tmem_wait_ld();
                    uint32_t pk[8];
                    if (sgc) {
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float s0v = __uint_as_float(rs[i]), s1v = __uint_as_float(rs[i + 1]);
                            const float d0 = __uint_as_float(rd[i]), d1 = __uint_as_float(rd[i + 1]);
                            const float g0 = gamma[(c % Ly::NG) * DK + c0 + i], g1 = gamma[(c % Ly::NG) * DK + c0 + i + 1];
                            const float a0 = g0 < kStrongGamma ? fmaf(s0v, g0, d0) : (s0v + d0) * g0;
                            const float a1 = g1 < kStrongGamma ? fmaf(s1v, g1, d1) : (s1v + d1) * g1;
                            pk[i / 2] = pack_bf16x2(a0, a1);
                            rs[i] = __float_as_uint(a0);
                            rs[i + 1] = __float_as_uint(a1);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            float a0 = __uint_as_float(rs[i]) + __uint_as_float(rd[i]);
                            float a1 = __uint_as_float(rs[i + 1]) + __uint_as_float(rd[i + 1]);
                            if (GATE) {
                                a0 *= gamma[(c % Ly::NG) * DK + c0 + i];
                                a1 *= gamma[(c % Ly::NG) * DK + c0 + i + 1];
                            }
                            pk[i / 2] = pack_bf16x2(a0, a1);
                            rs[i] = __float_as_uint(a0);
                            rs[i + 1] = __float_as_uint(a1);
                        }
                    }
                    tmem_st16(tS + c0, rs);
                    tmem_st8(tSB + c0 / 2, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_DS_EMPTY));
                    mbar_arrive(bar(B_S_READY + ((c + 1) & 1)));
                }
            }
            if (ok && !(GATE && !SAFE && *strong_flag)) {
                tc_fence_after();
                float* fs = (p.final_state && jl < jvalid) ? p.final_state + (long)bh * DK * dv + j : nullptr;
                const bool zl = norm && jl == 64 && p.final_z;
                for (int g = 0; g < COLS / 16; g++) {
                    uint32_t r[16];
                    tmem_ld16(tS + cbase + g * 16, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int d = cbase + g * 16 + i;
                        if (fs)
                            fs[(long)d * dv] = __uint_as_float(r[i]);
                        else if (zl)
                            p.final_z[(long)bh * DK + d] = __uint_as_float(r[i]);
                    }
                }
            }
        }
    } else if (warp < W_P0) {
        // ============================================================ output
        const int jl = lane_to_col<DVT>(warp & 3, lane);
        const bool store_col = jl >= 0 && jl < jvalid && !(norm && jl >= 64);
        const bool leader = warp == W_OUT0 && lane == 0;
        uint8_t* ost = sm + Ly::off_ost;
        for (int c = 0; c < N; c++) {
            bool ok = mbar_wait_warp(bar(B_O_FULL + (c & 1)), (c >> 1) & 1, abort_flag, p.err, p.wait_ns);
            // staging may be rewritten once the previous bulk store has read it
            if (leader && !p.out_f32) bulk_wait_group_read0();
            ok = bar_red_and(2, 128, ok);
            if (!ok) break;
            tc_fence_after();
            if (warp == W_OUT0 && lane == 0) GLA_TRACE_POINT(12, c);
            const int nval = min(C, L - c * C);
            if constexpr (DVT == 64) {
                // M = 64 rows sit in lanes 0-15 of each quarter: the 16x32bx2 shape gives
                // threads 0-15 tokens 0-31 and threads 16-31 tokens 32-63 of the same rows
                const int jr = lane_to_col<DVT>(warp & 3, lane & 15);
                const int t0 = (lane >> 4) * 32;
                uint32_t r[32];
                tmem_ld16x2_x32<32>(tmem + lane_field + kTmO + (c & 1) * 64, r);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_EMPTY + (c & 1)));
                if (jr < jvalid) {
                    if (!p.out_f32) {
                        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(ost) + jr + t0 * 64;
#pragma unroll
                        for (int t = 0; t < 32; t++) o[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]));
                    } else {
                        float* o = static_cast<float*>(p.out) + ((long)bh * L + (long)c * C + t0) * dv + j0 + jr;
#pragma unroll
                        for (int t = 0; t < 32; t++)
                            if (t0 + t < nval) o[(long)t * dv] = __uint_as_float(r[t]);
                    }
                }
            } else {
#pragma unroll 1
            for (int h = 0; h < 2; h++) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_field + kTmO + (c & 1) * 64 + h * 32, r);
                tmem_wait_ld();
                if (h == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_O_EMPTY + (c & 1)));
                }
                if (norm) {
                    if (jl == 64) {
#pragma unroll
                        for (int t = 0; t < 32; t++) den[h * 32 + t] = __uint_as_float(r[t]);
                    }
                    named_bar_sync(3, 128);
                }
                if (!store_col) continue;
                if (!p.out_f32) {
                    __nv_bfloat16* o =
                        reinterpret_cast<__nv_bfloat16*>(ost + (jl >> 6) * 8192) + (jl & 63) + h * 32 * 64;
                    if (norm) {
#pragma unroll
                        for (int t = 0; t < 32; t++) o[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]) / den[h * 32 + t]);
                    } else {
#pragma unroll
                        for (int t = 0; t < 32; t++) o[t * 64] = __float2bfloat16_rn(__uint_as_float(r[t]));
                    }
                } else {
                    float* o = static_cast<float*>(p.out) + ((long)bh * L + (long)c * C + h * 32) * dv + j0 + jl;
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float x = __uint_as_float(r[t]);
                        if (norm) x = x / den[h * 32 + t];
                        if (h * 32 + t < nval) o[(long)t * dv] = x;
                    }
                }
            }
            }
            if (!p.out_f32) {
                fence_proxy_async_smem();
                named_bar_sync(3, 128);
                if (leader) {
                    const int nblk = norm ? 1 : jvalid / 64;
                    for (int blk = 0; blk < nblk; blk++)
                        tma_store_3d(&p.tm_out, smem_u32(ost) + blk * 8192, j0 + blk * 64, c * C, bh);
                    bulk_commit_group();
                }
            }
            if (warp == W_OUT0 && lane == 0) GLA_TRACE_POINT(13, c);
        }
        if (leader && !p.out_f32) bulk_wait_group0();
    } else if (warp < W_TMA) {
        // ============================================================ P = tril(A) -> bf16
        const int t = threadIdx.x - W_P0 * 32;  // token row 0..63 (TMEM lanes 0..63)
        for (int c = 0; c < N; c++) {
            const int pb = c % Ly::NP;
            uint8_t* P = sm + Ly::off_p + pb * Ly::PB;
            if (!mbar_wait_warp(bar(B_A_FULL), c & 1, abort_flag, p.err, p.wait_ns)) break;
            if (!mbar_wait_warp(bar(B_P_EMPTY + pb), ((c / Ly::NP) & 1) ^ 1, abort_flag, p.err, p.wait_ns)) break;
            tc_fence_after();
            if (t == 0) GLA_TRACE_POINT(10, c);
            // strong channels of this chunk (published by the gate before the chunk's A product)
            uint32_t smask[4] = {0u, 0u, 0u, 0u};
            if constexpr (SAFE && GATE) {
                const volatile uint32_t* slot = ring + (c % kRing) * 5;
                if (!__all_sync(0xffffffffu, ring_wait(slot, static_cast<uint32_t>(c), abort_flag, p.err, p.wait_ns))) break;
                __threadfence_block();
#pragma unroll
                for (int e = 0; e < 4; e++) smask[e] = slot[1 + e];
            }
            if (SAFE && GATE && (smask[0] | smask[1] | smask[2] | smask[3]) != 0u) {
                const long row0 = (long)bh * L + (long)c * C;  // first token of the chunk in the raw inputs
                strong_scores<DK, SCALAR>(tmem + lane_field + TM_A, t, min(C, L - c * C),
                                          make_uint4(smask[0], smask[1], smask[2], smask[3]), p.q_raw + row0 * DK,
                                          p.k_raw + row0 * DK, p.la_raw + (SCALAR ? row0 : row0 * DK), elu);
            }
#pragma unroll 1
            for (int h = 0; h < 2; h++) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_field + TM_A + h * 32, r);
                tmem_wait_ld();
                if (h == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_A_EMPTY));
                    if (t == 0) GLA_TRACE_POINT(23, c);
                }

#pragma unroll
                for (int k8 = 0; k8 < 4; k8++) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int i = h * 32 + k8 * 8 + e;
                        x[e] = (i <= t) ? __uint_as_float(r[k8 * 8 + e]) : 0.f;
                    }
                    uint4 w;
                    w.x = pack_bf16x2(x[0], x[1]);
                    w.y = pack_bf16x2(x[2], x[3]);
                    w.z = pack_bf16x2(x[4], x[5]);
                    w.w = pack_bf16x2(x[6], x[7]);
                    *reinterpret_cast<uint4*>(P + sw128_offset(t, h * 32 + k8 * 8)) = w;
                }
            }
            if (t == 0) GLA_TRACE_POINT(15, c);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + pb));
            if (t == 0) GLA_TRACE_POINT(11, c);
        }
    } else if (warp == W_TMA) {
        // ============================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            if (GATE) tma_prefetch_desc(&p.tm_la);
            if (!p.out_f32) tma_prefetch_desc(&p.tm_out);
            // The three rings are refilled independently (a full V ring must not hold
            // back the next chunk's q/k and log alpha loads).
            // This thread also issues A(c) = Qh_c Kh_c^T: a tensor-core instruction costs
            // its issuing thread about as much as any other step of the MMA thread's
            // chunk, so the products are split between two issuers.
            constexpr uint32_t idA = make_idesc_bf16(128, 64, 0, 0);
            int na = 0;
            uint32_t idle = 0;
            unsigned long long t_last = 0;
            const int nl_end = GATE ? N : 0;
            while (pl_n < nl_end || pq_n < N || pv_n < N || na < N) {
                bool prog = false;
                // A(c) goes into the tensor pipe only after O_i(c-1): the state chain
                // waits on O_i(c-1), which must not queue behind A(c).
                if (na < pq_n && na <= *oi_issued && mbar_test(bar(B_QK_GATED + na % NS), (na / NS) & 1) &&
                    mbar_test(bar(B_A_EMPTY), (na & 1) ^ 1)) {
                    tc_fence_after();
                    GLA_TRACE_POINT(19, na);
                    const uint32_t Qs = sbase + Ly::off_qk + (na % NS) * Ly::STAGE_QK, Ks = Qs + Ly::QB;
                    // rows 64..127 of the M=128 tile read past the Q tile and are ignored
#pragma unroll
                    for (int kk = 0; kk < DK / 16; kk++) {
                        const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_ss(tmem + TM_A, make_sdesc(Qs + off, 16, 1024), make_sdesc(Ks + off, 16, 1024), idA,
                               kk > 0);
                    }
                    mma_commit(bar(B_A_FULL));
                    mma_commit(bar(B_QK_EMPTY + na % NS));
                    GLA_TRACE_POINT(9, na);
                    na++;
                    prog = true;
                }
                if (pl_n < nl_end && pl_n <= pq_n + 1 &&
                    mbar_test(bar(B_LA_EMPTY + pl_n % NL), ((pl_n / NL) & 1) ^ 1)) {
                    const int l = pl_n % NL;
                    mbar_arrive_expect_tx(bar(B_LA_FULL + l), Ly::LAB);
                    if (SCALAR)  // [B*H][L] fp32, box 64 tokens x 1
                        tma_load_3d(sbase + Ly::off_la + l * Ly::LAB, &p.tm_la, bar(B_LA_FULL + l), pl_n * C, bh, 0);
                    else
                        tma_load_3d(sbase + Ly::off_la + l * Ly::LAB, &p.tm_la, bar(B_LA_FULL + l), 0, pl_n * C, bh);
                    pl_n++;
                    prog = true;
                }
                if (pq_n < N && mbar_test(bar(B_QK_EMPTY + pq_n % NS), ((pq_n / NS) & 1) ^ 1)) {
                    const int s = pq_n % NS;
                    GLA_TRACE_POINT(1, pq_n);
                    mbar_arrive_expect_tx(bar(B_QK_FULL + s), 2 * Ly::QB);
                    const uint32_t qdst = sbase + Ly::off_qk + s * Ly::STAGE_QK;
                    for (int a = 0; a < DK / 64; a++) {
                        tma_load_3d(qdst + a * 8192, &p.tm_q, bar(B_QK_FULL + s), a * 64, pq_n * C, bh);
                        tma_load_3d(qdst + Ly::QB + a * 8192, &p.tm_k, bar(B_QK_FULL + s), a * 64, pq_n * C, bh);
                    }
                    pq_n++;
                    prog = true;
                }
                if (pv_n < N && mbar_test(bar(B_V_EMPTY + pv_n % NV), ((pv_n / NV) & 1) ^ 1)) {
                    const int v = pv_n % NV;
                    mbar_arrive_expect_tx(bar(B_V_FULL + v), nvb * 8192);
                    for (int blk = 0; blk < nvb; blk++)
                        tma_load_3d(sbase + Ly::off_v + v * Ly::VB + blk * 8192, &p.tm_v, bar(B_V_FULL + v),
                                    j0 + blk * 64, pv_n * C, bh);
                    pv_n++;
                    prog = true;
                }
                if (!prog) __nanosleep(20);
                if (prog) {
                    idle = 0;
                } else if ((++idle & 255u) == 0) {
                    if (*abort_flag) break;
                    const unsigned long long now = globaltimer();
                    if (idle == 256) {
                        t_last = now;
                    } else if (now - t_last > p.wait_ns) {
                        *abort_flag = 1;
                        record_timeout_code(p.err, 0x20000000u | ((pl_n & 0xff) << 16) | ((pq_n & 0xff) << 8) |
                                                       (pv_n & 0xff));
                        break;
                    }
                }
            }
            mma_commit(bar(B_DRAIN));
        }
    } else {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = make_idesc_bf16(DVT, DK, 1, 1);
            constexpr uint32_t idOi = make_idesc_bf16(DVT, 64, 0, 0);
            constexpr uint32_t idOa = make_idesc_bf16(DVT, 64, 1, 0);
            constexpr uint64_t kK = sdesc_const(16, 1024);     // K-major, 128-byte swizzle
            constexpr uint64_t kMN = sdesc_const(8192, 1024);  // MN-major, 64-column blocks 8 KB apart
            auto qs_of = [&](int c) { return sbase + Ly::off_qk + (c % NS) * Ly::STAGE_QK; };
            auto vs_of = [&](int c) { return sbase + Ly::off_v + (c % NV) * Ly::VB; };
            // chunk c's Qh/Kh are in its stage
            auto gated = [&](int c) { return mbar_test(bar(B_QK_GATED + c % NS), (c / NS) & 1); };
            // Issue each chunk's dS, O_i and O_a as soon as their inputs are ready (A is
            // the TMA thread's).  A phase that has completed stays complete until the
            // product waiting on it is issued, so each barrier is polled only until it
            // first passes.
            int nd = 0, ni = 0, no = 0, nq = 0;
            // 128-column tile: state updates known to be complete (chunks 0 .. ns-1); its
            // state warps read e^{b_C} from the q/k stage's slot and wait on the stage's gate
            // barrier, so a stage is released only after the chunk's state update
            int ns = 0;
            bool d_e = false, d_g = false, d_v = false;  // dS(nd): dS buffer free, gated, V landed
            bool i_s = false, i_o = false, i_g = false;  // O_i(ni): previous state's copy, O buffer free, gated
            unsigned long long t_last = globaltimer();
            uint32_t idle = 0;
            while (no < N) {
                bool prog = false;
                // dS(c) = V_c^T Kh_c first: the state chain waits on it.  64-column tile: dS(c)
                // lands in buffer c & 1, released by the state warps' read of dS(c - 2)
                if (nd < N) {
                    if (!d_e)
                        d_e = DVT == 64 ? mbar_test(bar(B_DS_EMPTY + (nd & 1)), ((nd >> 1) & 1) ^ 1)
                                        : mbar_test(bar(B_DS_EMPTY), nd & 1);
                    if (d_e && !d_g) d_g = gated(nd);
                    if (d_g && !d_v) d_v = mbar_test(bar(B_V_FULL + nd % NV), (nd / NV) & 1);
                    if (d_v) {
                        tc_fence_after();
                        const uint64_t vd = kMN | (vs_of(nd) >> 4), kd = kMN | ((qs_of(nd) + Ly::QB) >> 4);
#pragma unroll
                        for (int kk = 0; kk < C / 16; kk++)
                            mma_ss(tmem + (DVT == 64 ? (uint32_t)(nd & 1) * 128u : TM_DS), vd + kk * (2048 >> 4),
                                   kd + kk * (2048 >> 4), idS, kk > 0);
                        mma_commit(bar(B_DS_FULL + (DVT == 64 ? (nd & 1) : 0)));
                        nd++;
                        d_e = d_g = d_v = false;
                        prog = true;
                    }
                }
                // O_a(c) reads V(c): it goes only after dS(c), which this thread issued once
                // V(c) had landed (O_i(c) no longer implies that)
                if (no < ni && no < nd && mbar_test(bar(B_P_FULL + no % Ly::NP), (no / Ly::NP) & 1)) {
                    tc_fence_after();
                    const uint64_t vd = kMN | (vs_of(no) >> 4);
                    const uint64_t pd = kK | ((sbase + Ly::off_p + (no % Ly::NP) * Ly::PB) >> 4);
#pragma unroll
                    for (int kk = 0; kk < C / 16; kk++)
                        mma_ss(tmem + kTmO + (no & 1) * 64, vd + kk * (2048 >> 4), pd + kk * (32 >> 4), idOa, 1);
                    mma_commit(bar(B_O_FULL + (no & 1)));
                    mma_commit(bar(B_P_EMPTY + no % Ly::NP));
                    mma_commit(bar(B_V_EMPTY + no % NV));
                    no++;
                    prog = true;
                }
                if (ni < N) {
                    // the copy of the state before chunk ni (written after chunk ni - 1)
                    if (!i_s) i_s = mbar_test(bar(B_S_READY + (ni & 1)), (ni >> 1) & 1);
                    if (i_s && !i_o) i_o = mbar_test(bar(B_O_EMPTY + (ni & 1)), ((ni >> 1) & 1) ^ 1);
                    if (i_o && !i_g) i_g = gated(ni);
                    if (i_g) {
                        tc_fence_after();
                        // O^T = S^T Qh^T  (A operand: bf16 copy of the state before the chunk, in
                        // TMEM; Qh = q e^{b_t} carries the decay from the chunk start)
                        const uint64_t qd = kK | (qs_of(ni) >> 4);
                        // the copy: key channels 2x, 2x + 1 in column x
                        const uint32_t tsb = tmem + (DVT == 64 ? TM_CP64 : TM_SB);
#pragma unroll
                        for (int kk = 0; kk < DK / 16; kk++) {
                            const uint32_t off = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                            mma_ts(tmem + kTmO + (ni & 1) * 64, tsb + kk * 8, qd + off, idOi, kk > 0);
                        }
                        // the copy takes the next state once O_i(ni) has read it
                        mma_commit(bar(B_SB_EMPTY));
                        ni++;
                        *oi_issued = ni;
                        i_s = i_o = i_g = false;
                        if (ns < ni - 1) ns = ni - 1;  // O_i(c) read the state after chunk c - 1
                        prog = true;
                    }
                }
                // state(ns) complete: its S_READY phase (no later phase of that barrier can have
                // completed: the state warps' next update there waits on O_i(ns + 1), not issued)
                if (DVT == 128 && ns < nd && mbar_test(bar(B_S_READY + ((ns + 1) & 1)), ((ns + 1) >> 1) & 1)) {
                    ns++;
                    prog = true;
                }
                // this thread's share of the release of chunk nq's q/k stage: its dS and O_i
                // have finished (O_i(nq) may go before dS(nq)), and with the 128-column tile
                // the state update of nq (the TMA thread releases its A)
                while (nq < ni && nq < nd && (DVT == 64 || nq < ns)) {
                    mma_commit(bar(B_QK_EMPTY + nq % NS));
                    nq++;
                }
                if (!prog) __nanosleep(20);
                if (prog) {
                    idle = 0;
                } else if ((++idle & 255u) == 0) {
                    if (*abort_flag) break;
                    const unsigned long long now = globaltimer();
                    if (idle == 256) t_last = now;
                    else if (now - t_last > p.wait_ns) {
                        *abort_flag = 1;
                        // scheduler progress at the time: next dS, stage release, O_i, O_a chunk
                        record_timeout_code(p.err, 0x40000000u | ((nd & 0xff) << 22) | ((nq & 0xff) << 14) |
                                                       ((ni & 0xff) << 6) | ((no & 0x1f) << 1));
                        break;
                    }
                }
            }
            // drain: every issued tcgen05 op has finished before TMEM is released
            mma_commit(bar(B_DRAIN));
            volatile int no_abort = 0;
            mbar_wait(bar(B_DRAIN), 0, &no_abort, p.err);
        }
    }

    // ---------------------------------------------------------------- teardown
    if (warp == W_TMA && lane == 0 && *abort_flag) {
        // wait (bounded) for loads that may still be in flight
        volatile int no_abort = 0;
        for (int c = max(0, pq_n - NS); c < pq_n; c++) mbar_wait(bar(B_QK_FULL + c % NS), (c / NS) & 1, &no_abort, p.err);
        for (int c = max(0, pv_n - NV); c < pv_n; c++) mbar_wait(bar(B_V_FULL + c % NV), (c / NV) & 1, &no_abort, p.err);
        for (int c = max(0, pl_n - NL); c < pl_n; c++) mbar_wait(bar(B_LA_FULL + c % NL), (c / NL) & 1, &no_abort, p.err);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // every role has finished and every copy has landed: the exact pass may reuse the CTA
    return GATE && !SAFE && *strong_flag && !*abort_flag;
}

// The exact pass as a function of its own: its code and register allocation stay
// out of the pass that every call runs.
template <int DK, int DVT, bool SCALAR>
__device__ __noinline__ void exact_pass(const TcParams& p, uint8_t* smem_raw) {
    prefill_pass<DK, DVT, true, SCALAR, true>(p, smem_raw);
}

template <int DK, int DVT, bool GATE, bool SCALAR>
__global__ void __launch_bounds__(kThreads, 1) gla_prefill_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const bool redo = prefill_pass<DK, DVT, GATE, SCALAR, false>(p, smem_raw);
    if constexpr (GATE) {
        if (redo) exact_pass<DK, DVT, SCALAR>(p, smem_raw);
    }
    if ((threadIdx.x >> 5) == W_MMA) {
        const uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
        tc_fence_after();
        tmem_dealloc(*reinterpret_cast<const uint32_t*>(sm + Layout<DK, DVT, SCALAR>::off_misc), TM_COLS);
    }
}

CUresult encode_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int d0, int d1, int d2,
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

template <int DK, int DVT, bool GATE, bool SCALAR>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    if (encode_3d(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, DK, a.L, BH, 64, C, CU_TENSOR_MAP_SWIZZLE_128B) !=
            CUDA_SUCCESS ||
        encode_3d(&p.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, DK, a.L, BH, 64, C, CU_TENSOR_MAP_SWIZZLE_128B) !=
            CUDA_SUCCESS ||
        encode_3d(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, a.dv, a.L, BH, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (GATE && !SCALAR &&
        encode_3d(&p.tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.log_alpha, DK, a.L, BH, DK, C,
                  CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // one log alpha per token: [B*H][L] (row stride L*4 bytes, a multiple of 16 when L % 4 == 0)
    if (GATE && SCALAR &&
        encode_3d(&p.tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.log_alpha, a.L, BH, 1, C, 1,
                  CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.out_f32 = a.out_dtype == GLA_DTYPE_F32;
    if (!p.out_f32 && encode_3d(&p.tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, a.dv, a.L, BH, 64, C,
                                CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.q_raw = static_cast<const uint16_t*>(a.q);
    p.k_raw = static_cast<const uint16_t*>(a.k);
    p.la_raw = a.log_alpha;
    p.init_state = a.init_state;
    p.init_z = a.init_z;
    p.out = a.out;
    p.final_state = a.final_state;
    p.final_z = a.final_z;
    p.err = a.err_word;
    p.wait_ns = a.wait_ns;
    p.test_stall = a.test_stall;
    p.L = a.L;
    p.dv = a.dv;
    p.nchunks = (a.L + C - 1) / C;
    p.ntile = (a.dv + DVT - 1) / DVT;
    p.flags = a.flags;
    auto kern = gla_prefill_tc_kernel<DK, DVT, GATE, SCALAR>;
    const int smem = Layout<DK, DVT, SCALAR>::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long grid = (long)BH * p.ntile;
    kern<<<dim3((unsigned)grid), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// Value-tile width: 128 columns unless that leaves too few CTAs to cover the
// GPU's SMs, in which case 64 (twice the CTAs, M = 64 MMAs).
// GLA_TC_DVT=64|128 in the environment forces the width (used by the tests to
// cover both kernel variants on small shapes).
int choose_dvt(const PrefillArgs& a) {
    if (a.flags & GLA_FLAG_NORMALIZE) return 128;  // the normaliser column needs a spare lane
    if (const char* e = getenv("GLA_TC_DVT")) {
        if (e[0] == '6') return 64;
        if (e[0] == '1') return 128;
    }
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long ctas128 = (long)a.B * a.H * ((a.dv + 127) / 128);
    return ctas128 * 4 < (long)sms * 3 ? 64 : 128;
}

template <int DK, int DVT>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t s) {
    if (!a.log_alpha) return launch_t<DK, DVT, false, false>(a, s);
    return (a.flags & GLA_FLAG_SCALAR_GATE) ? launch_t<DK, DVT, true, true>(a, s) : launch_t<DK, DVT, true, false>(a, s);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
    if (a.in_dtype != GLA_DTYPE_BF16) return false;
    if (a.flags & GLA_FLAG_FORCE_SIMT) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv < 64 || a.dv % 64 != 0) return false;
    if ((a.flags & GLA_FLAG_NORMALIZE) && a.dv != 64) return false;
    if (a.L < 1) return false;
    // the per-token gate's tensor map needs a 16-byte row stride
    if (a.log_alpha && (a.flags & GLA_FLAG_SCALAR_GATE) && a.L % 4 != 0) return false;
    const long grid = (long)a.B * a.H * (a.dv / 64);
    if (grid > INT_MAX) return false;
    return true;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
    const int dvt = choose_dvt(a);
    if (a.dk == 64) return dvt == 64 ? launch_g<64, 64>(a, s) : launch_g<64, 128>(a, s);
    return dvt == 64 ? launch_g<128, 64>(a, s) : launch_g<128, 128>(a, s);
}

}  // namespace gla
