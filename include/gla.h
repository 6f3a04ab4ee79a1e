/*
 * gla.h -- C ABI of the GB300 (sm_103a) causal gated-linear-attention library.
 *
 * The operation (sources are the pages' titles and sections):
 *
 *   "Gated Linear Attention" (garden note), GLA Recurrent Form, eq. block:
 *       S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T,   alpha_t in (0,1)^{d_k},
 *   and its flowchart: o_t is q_t applied to the updated state, o_t = S_t^T q_t.
 *   "linear-attention" blog, Linear attention: the fixed-size state replaces
 *   the KV cache, o_n = o_n(S_{n-1}, q_n, k_n, v_n); with alpha == 1 the state
 *   is a running sum of k_i v_i^T (section Prefill).
 *   "Gated Linear Attention", Summary / Chunk-Wise Block-Parallel: prefill
 *   evaluates the same function chunk by chunk, O(L C d + L d^2).
 *   "Transformers are RNNs" notes, kernel derivation: optional feature map
 *   phi and normalised form o_t = phi(q_t)^T S_t / phi(q_t)^T z_t.
 *
 * Conventions of this library:
 *   - S is d_k x d_v (rows = key channels, decayed by alpha; columns = value
 *     channels), stored fp32 row-major per (batch, head).
 *   - Inputs are head-major: q, k, log_alpha [B][H][L][d_k]; v, out
 *     [B][H][L][d_v]; states [B][H][d_k][d_v].  All contiguous.
 *   - log_alpha is the natural log of the gate (fp32, finite, <= 0, i.e.
 *     alpha in (0, 1]); the library never applies a sigmoid or a temperature:
 *     the caller passes log alpha.  Every such gate is computed exactly, with
 *     no lower bound on alpha ("Gated Linear Attention", GLA Recurrent Form).
 *     On the tensor-core path a chunk over which some key channel decays by
 *     more than e^-64 makes its CTA compute its (head, value slice) a second
 *     time with that channel's intra-chunk scores evaluated with exponents
 *     <= 0 -- exact, but slower for such slices.
 *   - phi(x) = elu(x) + 1 when GLA_FLAG_FEATURE_ELU1 is set; the normaliser
 *     z (GLA_FLAG_NORMALIZE) is carried like one extra all-ones value column
 *     of the state, so it is decayed by alpha exactly like S.
 *
 * Ownership and threading: every pointer is caller-owned DEVICE memory
 * (16-byte aligned).  The library allocates no memory and holds no state
 * between calls except one device-side error word (see gla_device_error);
 * calls are asynchronous on the caller's stream.
 *
 * Errors: argument validation happens on the host before any launch and
 * returns a non-zero gla_status without touching the GPU.  Launch failures
 * return GLA_ERR_CUDA.  Device-side pipeline waits are bounded; a wait that
 * runs out sets the device error word (GLA_ERR_TIMEOUT) and the kernel
 * returns early, leaving the outputs undefined.  With the environment
 * variable GLA_SYNC_CHECK=1 every call synchronises its stream and reports
 * both kinds of error directly.
 */
#ifndef GLA_H
#define GLA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GLA_OK = 0,
    GLA_ERR_INVALID = 1,      /* NULL where required, negative size, out/in alias */
    GLA_ERR_UNSUPPORTED = 2,  /* shape/dtype/chunk combination not implemented */
    GLA_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    GLA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, ...) */
    GLA_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out */
} gla_status;

enum { GLA_DTYPE_BF16 = 0, GLA_DTYPE_F32 = 1 };

enum {
    GLA_FLAG_FEATURE_ELU1 = 1u,  /* apply phi(x) = elu(x) + 1 to q and k */
    GLA_FLAG_NORMALIZE = 2u,     /* o_t = phi(q_t)^T S_t / phi(q_t)^T z_t */
    GLA_FLAG_FORCE_SIMT = 4u,    /* use the fp32 SIMT chunk kernel even for bf16 */
    GLA_FLAG_FORCE_CHUNK = 8u,   /* use a chunk kernel even for a sequence of <= 16 tokens */
    GLA_FLAG_SCALAR_GATE = 16u   /* log_alpha is fp32 [B][H][L]: one gate per token, shared by all
                                    key channels ("Gated Linear Attention", the scalar special case
                                    of the gate matrix G_t = alpha_t 1^T with alpha_t = gamma_t 1) */
};

/*
 * gla_fwd -- chunk-wise prefill ("Gated Linear Attention", Chunk-Wise
 * Block-Parallel; recurrence from GLA Recurrent Form).
 *
 *   q, k        bf16 [B][H][L][dk]
 *   v           bf16 [B][H][L][dv]
 *   log_alpha   fp32 [B][H][L][dk], or NULL for alpha == 1 (plain linear attention)
 *   init_state  fp32 [B][H][dk][dv], or NULL for S_{-1} = 0
 *   out         bf16 [B][H][L][dv]  (o_t = S_t^T q_t, inclusive of token t)
 *   final_state fp32 [B][H][dk][dv], or NULL; may alias init_state
 *   chunk       chunk length C; must be 64
 *   stream      cudaStream_t (NULL = legacy default stream)
 * Supported: dk in {64, 128}, dv a multiple of 64 (tensor-core kernel); any
 * other dk, dv in [1, 256] runs on the SIMT kernel.  L >= 0, B, H >= 1.
 * A call of 1..16 tokens (the prefill-to-decode hand-off: several new tokens
 * per sequence on top of init_state) runs the recurrence token by token in
 * fp32 on a kernel that reads and writes each head's state once, when
 * dk % 16 == 0, dv % 4 == 0 and 2048 <= dk*dv <= 32768 with dk*dv a multiple
 * of 2048 (no feature map or normaliser); GLA_FLAG_FORCE_CHUNK turns this off.
 * out must not alias any input.
 */
int gla_fwd(const void* q, const void* k, const void* v, const float* log_alpha,
            const float* init_state, void* out, float* final_state,
            int B, int H, int L, int dk, int dv, int chunk, void* stream);

/* Extended prefill arguments (same layouts as gla_fwd). */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;     /* NULL: alpha == 1 */
    const float* init_state;    /* NULL: zero */
    const float* init_z;        /* [B][H][dk], NORMALIZE only; NULL: zero */
    void* out;
    float* final_state;         /* NULL: not written */
    float* final_z;             /* [B][H][dk], NORMALIZE only; NULL: not written */
    int B, H, L, dk, dv, chunk;
    int in_dtype;               /* GLA_DTYPE_BF16 or GLA_DTYPE_F32 (q, k, v) */
    int out_dtype;              /* GLA_DTYPE_BF16 or GLA_DTYPE_F32 */
    unsigned flags;             /* GLA_FLAG_* */
} gla_fwd_args;

/*
 * gla_fwd_ex -- gla_fwd with input/output dtypes, feature map, normaliser and
 * the normaliser state.  fp32 inputs run on the SIMT kernel in exact fp32
 * arithmetic (no TF32).  Same validation and error behaviour as gla_fwd.
 */
int gla_fwd_ex(const gla_fwd_args* a, void* stream);

/*
 * gla_fwd_host -- gla_fwd_ex on host-resident data, with the host<->device
 * copies overlapped with the computation.  The (batch, head) pairs are
 * independent problems ("Gated Linear Attention", GLA Recurrent Form: each
 * head carries its own state), so they are split into `groups` contiguous
 * groups; group g's inputs are copied host->device on `copy_in`, computed on
 * `compute` once they have landed, and its outputs copied device->host on
 * `copy_out` once computed, so the copies of one group overlap the kernels and
 * the copies of the others.
 *
 *   host    gla_fwd_args of HOST pointers (page-locked for the copies to be
 *           asynchronous): inputs q, k, v, log_alpha, init_state, init_z;
 *           outputs out, final_state, final_z.
 *   dev     gla_fwd_args of caller-owned DEVICE buffers with the same shapes
 *           (the staging area), same B, H, L, dk, dv, chunk, dtypes and flags;
 *           each buffer given on both sides or on neither; final_state (and
 *           final_z) must not alias init_state (init_z) here.
 *   groups  >= 1.  Group boundaries fall on multiples of the smallest head
 *           count whose bytes in every buffer are a multiple of 16 (so each
 *           group's slices stay 16-byte aligned); more groups than that allows
 *           are clamped.
 * Ordering: the call first makes `copy_in` wait for work already queued on
 * `compute` and `compute` wait for work already queued on `copy_out`, so
 * back-to-back calls reuse the staging area safely.  The call returns once
 * everything is queued; the host outputs are complete when `copy_out` has
 * drained.  Events it needs are created and released by the call.  Validation
 * failures return before anything is queued.
 */
int gla_fwd_host(const gla_fwd_args* host, const gla_fwd_args* dev, int groups, void* copy_in, void* compute,
                 void* copy_out);

/*
 * gla_decode_step -- one recurrent step per (sequence, head) ("linear-attention"
 * blog, Linear attention: o_n from S_{n-1}, q_n, k_n, v_n; gate from GLA
 * Recurrent Form).
 *
 *   q, k       bf16 [B][H][dk]     (one token per sequence)
 *   v          bf16 [B][H][dv]
 *   log_alpha  fp32 [B][H][dk], or NULL for alpha == 1
 *   state      fp32 [B][H][dk][dv], updated IN PLACE: S <- Diag(alpha) S + k v^T
 *   out        fp32 [B][H][dv]: o = S_new^T q
 * Supported: dv a multiple of 4, dv <= 512, dk in [1, 512].  out must not alias.
 */
int gla_decode_step(const void* q, const void* k, const void* v, const float* log_alpha,
                    float* state, float* out, int B, int H, int dk, int dv, void* stream);

/*
 * gla_delta_fwd -- the delta rule ("linear-attention" blog, Delta attention):
 * before each write the memory's prediction for the key is taken and only the
 * error is written, with strength beta_n; the gated variant decays the state
 * first ("Gated Linear Attention", GLA Recurrent Form):
 *   S <- Diag(alpha_n) S;  p = S^T k_n;  u = beta_n (v_n - p);  S <- S + k_n u^T;
 *   o_n = S^T q_n.
 *
 *   q, k        bf16 [B][H][L][dk]
 *   v           bf16 [B][H][L][dv]
 *   beta        fp32 [B][H][L]  (write strength per token)
 *   log_alpha   fp32 [B][H][L][dk], or NULL for no gate
 *   init_state  fp32 [B][H][dk][dv], or NULL for S_{-1} = 0
 *   out         [B][H][L][dv], bf16 or fp32 (out_dtype = GLA_DTYPE_BF16 / _F32)
 *   final_state fp32 [B][H][dk][dv], or NULL; may alias init_state
 * With d_k = d_v = 128 it runs in chunk form on the tensor cores (see
 * gla_delta_fwd_ex); otherwise the recurrence runs token by token in fp32.
 * Supported: dk in {32, 64, 128}, dv a multiple of 16.  Pointers 16-byte
 * aligned; out must not alias an input.
 * Validation failures return before any launch.
 */
int gla_delta_fwd(const void* q, const void* k, const void* v, const float* beta, const float* log_alpha,
                  const float* init_state, void* out, float* final_state, int B, int H, int L, int dk, int dv,
                  int out_dtype, void* stream);

/*
 * gla_delta_fwd_ex -- gla_delta_fwd with flags (0 or GLA_FLAG_FORCE_SIMT).
 *
 * With d_k = d_v = 128 the delta rule runs in chunk form on the tensor cores
 * ("linear-attention" blog, Delta attention / Prefill: the writes of a chunk
 * solve one unit lower-triangular system): per chunk of 64 tokens, with
 * A = (k e^{b_t-b_C}) (k e^{b_C-b_i})^T, T = (I + Diag(beta) tril_strict(A))^{-1}
 * and M = T Diag(beta), the writes are U = M (V - Kr S') and
 * o = Qh S' + tril(Qh Kh^T) U, S_C = S' + Kh^T U (bf16 tensor-core products,
 * fp32 accumulation and state; T in fp32).  Heads with a chunk over which a
 * channel decays by more than e^-64 are recomputed by the token-by-token
 * kernel, which also serves every other shape and GLA_FLAG_FORCE_SIMT.
 * Same arguments, validation and error behaviour as gla_delta_fwd.
 */
int gla_delta_fwd_ex(const void* q, const void* k, const void* v, const float* beta, const float* log_alpha,
                     const float* init_state, void* out, float* final_state, int B, int H, int L, int dk, int dv,
                     int out_dtype, unsigned flags, void* stream);

/*
 * gla_bwd -- gradients of the recurrence ("Gated Linear Attention", GLA
 * Recurrent Form: S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t)
 * for a loss L with dout = dL/do_t and dfinal = dL/dS_{L-1}.  With
 * G_t = dL/dS_t = Diag(alpha_{t+1}) G_{t+1} + q_t dout_t^T:
 *   dq_t = S_t dout_t,  dk_t = G_t v_t,  dv_t = G_t^T k_t,
 *   dinit = Diag(alpha_0) G_0,
 *   dlog_alpha_t = sum_{s >= t} (q_s * dq_s - k_s * dk_s) + rowsum(dfinal * S_{L-1})
 *     (the gate enters only through its cumulative sums, so this equals
 *      alpha_t * rowsum(G_t * S_{t-1})).
 *
 *   q, k        [B][H][L][dk], bf16 or fp32 (in_dtype)
 *   v, dout     [B][H][L][dv], in_dtype
 *   log_alpha   fp32 [B][H][L][dk], or NULL for no gate; [B][H][L] with
 *               GLA_FLAG_SCALAR_GATE (one gate per token, all channels)
 *   init_state  fp32 [B][H][dk][dv], or NULL for S_{-1} = 0
 *   dfinal      fp32 [B][H][dk][dv], or NULL for dL/dS_{L-1} = 0
 *   dq, dk_out  fp32 [B][H][L][dk]      (written)
 *   dv_out      fp32 [B][H][L][dv]      (written)
 *   dlog_alpha  fp32 [B][H][L][dk], or NULL (needs log_alpha); [B][H][L]
 *               with GLA_FLAG_SCALAR_GATE: the sum of the per-channel
 *               gradients, accumulated across row blocks with fp32 atomics
 *               (the order of that sum is not fixed)
 *   dinit       fp32 [B][H][dk][dv], or NULL
 *   flags       0 or GLA_FLAG_SCALAR_GATE
 * All caller-owned device memory, 16-byte aligned; outputs must not overlap
 * inputs or each other.  The recurrence runs token by token in fp32 (one
 * launch: row blocks sweep forward for dq, then backward for dk, dlog_alpha
 * and dinit; column blocks sweep backward for dv).  Supported: dk, dv in
 * {32, 64, 128}.  Validation failures return before any launch; L = 0 only
 * writes dinit (= dfinal, or zero).
 */
int gla_bwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* init_state,
            const void* dout, const float* dfinal, float* dq, float* dk_out, float* dv_out, float* dlog_alpha,
            float* dinit, int B, int H, int L, int dk, int dv, int in_dtype, unsigned flags, void* stream);

/*
 * gla_device_error -- synchronise `stream`, read and clear the device error
 * word that bounded waits set.  Returns GLA_OK, GLA_ERR_TIMEOUT or GLA_ERR_CUDA.
 * The record is one per device and process, shared by every call on every
 * stream: a wait that ran out in a call on one stream is reported to (and
 * cleared by) whichever caller reads the record next, on any stream.  Callers
 * that run concurrent calls on several streams should read it only after
 * synchronising all of them.
 */
int gla_device_error(void* stream);

/*
 * gla_device_error_detail -- synchronise `stream` and copy (without clearing)
 * the device error record into detail4[4]: [0] flags (bit 0 = a bounded wait
 * timed out), [1] the first timed-out wait (shared-memory barrier address,
 * bit 31 = awaited parity, bit 0 set; bit 30 set = the MMA issuer's
 * readiness loop, with its chunk counters in bits 1-29; bit 29 set = the TMA
 * producer's loop, with its chunk counters in bits 0-23), [2] thread index,
 * [3] CTA index.  For diagnosing a GLA_ERR_TIMEOUT; gla_device_error clears it.
 */
int gla_device_error_detail(void* stream, unsigned* detail4);

/*
 * gla_test_set_waits -- TEST ONLY.  For the calls that follow: `limit_ns` is
 * the limit, in nanoseconds, of the tensor-core prefill kernel's pipeline
 * waits (0 restores the default of 2 s; the waits that drain copies and
 * products still in flight before a CTA exits always keep the default), and
 * with `stall` nonzero the kernel's gate role first waits on a barrier that
 * nothing completes, so that wait runs out after `limit_ns`, every role of the
 * CTA stops, and the call reports GLA_ERR_TIMEOUT through gla_device_error
 * (outputs undefined).  Used to check the error path and that the device stays
 * usable afterwards.  Process-wide; not thread-safe.  Returns GLA_OK.
 *
 * Also for tests: with GLA_TEST_FAIL_LAUNCH=1 in the environment, every entry
 * point that launches a kernel returns GLA_ERR_CUDA after its argument
 * validation and before any launch (an injected launch failure).
 */
int gla_test_set_waits(unsigned long long limit_ns, int stall);

/* Human-readable name of a gla_status value (static string). */
const char* gla_status_string(int status);

/* Library version string (static). */
const char* gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H */
