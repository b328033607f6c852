/*
 * pi_attn.h -- C ABI of the GB300 (sm_103a) pi-Attention / ECP attention library.
 *
 * Operation.  For every batch b, query head h and query position i, one
 * softmax runs over the union U(i) of two key sets, and the output is the
 * softmax-weighted sum of the value rows:
 *
 *   pi mode ("pi-Attention: Periodic Sparse Transformers for Efficient
 *   Long-Context Modeling", section 2 "Methodology"):
 *     L(i) = { j : max(0, i - k_local) <= j <= i }          (2.1 ring-local band,
 *                                                           causal, both ends kept)
 *     P(i) = { i - m*period : m = 1..S, i - m*period >= 0,
 *              m*period > k_local }                        (2.2 pi-skip keys,
 *                                                           causal; a skip key
 *                                                           already in the band is
 *                                                           not repeated)
 *     z_ij = (q_i . k_j) / sqrt(d) + ln(alpha_i)     for j in L(i)
 *     z_ij = (q_i . k_j) / sqrt(d) + ln(1 - alpha_i) for j in P(i)   (2.3 gate as
 *                                                           log-prior, one softmax
 *                                                           over the union)
 *   bidirectional pi mode (the same page, 2.1 and 2.2 in their general,
 *   non-causal form; forward and backward):
 *     L(i) = { j : max(0, i - k_local) <= j <= min(N - 1, i + k_local) }
 *     P(i) = { i - m*period : i - m*period >= 0 } u { i + m*period : i + m*period < N },
 *            m = 1..S with m*period > k_local,   priors as in pi mode
 *   ECP mode ("Efficient Context Propagating Perceiver Architectures for
 *   Auto-Regressive Language Modeling", section 2, paired-segment PAR block):
 *     with half-segment length c = k_local and s = floor(i / c):
 *     U(i) = { j : max(0, (s - 1) * c) <= j <= i },  z_ij = (q_i . k_j) / sqrt(d)
 *   GQA (attention branch of the GSS-Transformer hybrid page): query head h
 *   reads key/value head floor(h / (H / Hkv)).
 *
 *   lse_i = ln sum_{j in U(i)} exp(z_ij);  out_i = sum_j exp(z_ij - lse_i) v_j.
 *   A row with no finite logit (alpha_i = 0 and P(i) empty) gets out_i = 0 and
 *   lse_i = -inf.
 *
 * Layouts (all contiguous, row-major, element strides implied by the shape):
 *   q, out, dq, dout : [B, H,   N, d]
 *   k, v, dk, dv     : [B, Hkv, N, d]
 *   alpha, lse, dalpha : [B, H, N] fp32
 * "bf16" entry points take bfloat16 q/k/v/out/dout/dq/dk/dv; "_f32" entry
 * points take fp32.  alpha, lse and dalpha are always fp32.
 *
 * Ownership.  The caller owns every buffer and the stream.  The library never
 * allocates per call; the only device state it keeps is one int status word
 * per device, a static device variable.
 *
 * Asynchrony.  Every compute entry point only enqueues work on `stream`
 * (a cudaStream_t passed as void*, NULL = legacy default stream) and returns
 * PI_OK once the kernels are launched.  Device-side failures (a bounded wait
 * that ran out) are reported later by pi_attn_status().
 *
 * Validation.  Every argument is checked before anything is launched; a bad
 * argument returns a negative pi_status_t and launches nothing:
 *   PI_ERR_NULL        a required pointer is NULL (alpha may be NULL only in
 *                      ECP mode, where it is unused)
 *   PI_ERR_SHAPE       B, H, Hkv, N <= 0; H % Hkv != 0; k_local < 0; S < 0;
 *                      period <= 0 while S > 0; ECP with k_local <= 0 or S != 0
 *   PI_ERR_UNSUPPORTED d not in {32, 64, 128}; unknown mode; sizes whose
 *                      element offsets overflow int64 or whose row count
 *                      exceeds 2^31-1; (debug calls) N above their limit
 *   PI_ERR_ALIGN       a bf16/fp32 tensor of shape [.., d] not 16-byte aligned,
 *                      or an fp32 vector (alpha, lse, dalpha) not 4-byte aligned
 *   PI_ERR_WORKSPACE   backward workspace NULL or smaller than required
 *   PI_ERR_CUDA        a CUDA runtime error at launch (cudaGetLastError)
 *   PI_ERR_DEVICE_TIMEOUT  (from pi_attn_status) a device-side bounded wait
 *                      gave up; the kernel returned without finishing.  The
 *                      status word is sticky: until pi_attn_status() reads and
 *                      clears it, later launches on that device give up at their
 *                      first wait that is not already satisfied, so their
 *                      outputs are undefined.
 */
#ifndef PI_ATTN_H_
#define PI_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PI_MODE_PI = 0, PI_MODE_ECP = 1, PI_MODE_PI_BIDIR = 2 } pi_mode_t;

typedef enum {
    PI_OK = 0,
    PI_ERR_NULL = -1,
    PI_ERR_SHAPE = -2,
    PI_ERR_UNSUPPORTED = -3,
    PI_ERR_ALIGN = -4,
    PI_ERR_WORKSPACE = -5,
    PI_ERR_CUDA = -6,
    PI_ERR_DEVICE_TIMEOUT = -7
} pi_status_t;

/*
 * pi_attn_fwd -- fused sparse causal attention forward, bf16 in/out, fp32
 * accumulation (pi-Attention section 2.1-2.3; ECP section 2).
 *   q [B,H,N,d], k/v [B,Hkv,N,d] bf16 (device); alpha [B,H,N] fp32 (device,
 *   values in [0,1]; may be NULL in ECP mode); k_local = band width k (pi
 *   mode) or half-segment length c (ECP mode); period = skip stride pi;
 *   S = number of skip multiples (0 = band only); mode = pi_mode_t.
 *   Writes out [B,H,N,d] bf16 (round-to-nearest-even) and lse [B,H,N] fp32
 *   (natural log).  d = 64 and 128 run on the tcgen05/TMEM/TMA kernel; d = 32
 *   runs on the CUDA-core kernel.  Deterministic.
 */
int pi_attn_fwd(const void *q, const void *k, const void *v, const float *alpha,
                int B, int H, int Hkv, int N, int d, int k_local, int period, int S, int mode,
                void *out, float *lse, void *stream);

/* pi_attn_fwd_f32 -- same operation and arguments with fp32 q/k/v/out (CUDA-core
 * kernel, fp32 throughout).  Deterministic. */
int pi_attn_fwd_f32(const void *q, const void *k, const void *v, const float *alpha,
                    int B, int H, int Hkv, int N, int d, int k_local, int period, int S,
                    int mode, void *out, float *lse, void *stream);

/*
 * pi_attn_fwd_gated -- pi_attn_fwd with the gate fused into the same launch
 * ("pi-Attention" page, section 2.3: a light neural network (MLP) produces alpha
 * per token and per head from the input content).  Reading of the network: one
 * hidden layer of PI_ATTN_GATE_HIDDEN units with a ReLU on the head's query, and
 * a logistic output:
 *     hid_f = max(0, sum_t gate_w1[h][f][t] q_{b,h,i,t} + gate_b1[h][f]),
 *     alpha_{b,h,i} = 1 / (1 + exp(-(sum_f gate_w2[h][f] hid_f + gate_b2[h]))),
 * computed with the hidden pre-activations W1_h q on the tensor core (the block's query tile times the
 * W1 rows of its heads, bf16 operands, fp32 accumulation; one extra key tile per block), the
 * rest in fp32, then used exactly as pi_attn_fwd uses its alpha input.
 *   gate_w1 [H, PI_ATTN_GATE_HIDDEN, d] bf16 (16-byte aligned), gate_b1 and gate_w2
 *   [H, PI_ATTN_GATE_HIDDEN] fp32, gate_b2 [H] fp32; alpha_out [B, H, N] fp32 (may be
 *   NULL; receives the gate's alpha, e.g. for pi_attn_bwd, whose dalpha is then the
 *   gradient with respect to these values; the gate's own weight gradients follow
 *   from it by the chain rule on the caller's side).  mode: pi or bidirectional
 *   (ECP: PI_ERR_UNSUPPORTED); d: 64 or 128 (else PI_ERR_UNSUPPORTED).  Other
 *   arguments, layouts and errors as pi_attn_fwd.
 */
#define PI_ATTN_GATE_HIDDEN 8
int pi_attn_fwd_gated(const void *q, const void *k, const void *v, const void *gate_w1,
                      const float *gate_b1, const float *gate_w2, const float *gate_b2, int B,
                      int H, int Hkv, int N, int d, int k_local, int period, int S, int mode,
                      void *out, float *lse, float *alpha_out, void *stream);

/*
 * pi_attn_bwd_workspace_size -- bytes of device workspace pi_attn_bwd needs
 * for these sizes: one fp32 per query row for D_i = sum_j p_ij (dout_i . v_j),
 * which equals dout_i . out_i in exact arithmetic; it is recomputed from the
 * probabilities rather than read from the bf16-rounded out.
 */
size_t pi_attn_bwd_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * pi_attn_bwd -- backward of pi_attn_fwd (the chain rule through the
 * definition above; bf16 tensors, fp32 accumulation).
 *   Inputs: q, k, v, alpha as for the forward; out [B,H,N,d] and lse [B,H,N]
 *   from pi_attn_fwd; dout [B,H,N,d].  D_i is recomputed exactly from the
 *   probabilities; out only supplies dout_i . out_i, a per-row centre that keeps
 *   the bf16 operands of the dq accumulation small (any out gives the same
 *   result up to rounding).
 *   Outputs: dq [B,H,N,d], dk and dv [B,Hkv,N,d] (summed over the query heads
 *   of each KV group) bf16; dalpha [B,H,N] fp32 (may be NULL; zero in ECP mode),
 *   computed as dalpha_i = -(sum_{j in P(i)} dz_ij) / (alpha_i (1 - alpha_i)),
 *   which equals sum_L dz/alpha - sum_P dz/(1-alpha) because every softmax row
 *   of dz sums to zero; where alpha_i is exactly 0 or 1 (one prior is -inf, a
 *   saturated gate) dalpha_i is 0, so that a gate whose fp32 sigmoid rounds to
 *   1 passes no NaN upstream.  dz_ij = p_ij (dout_i . v_j - D_i),
 *   D_i = sum_j p_ij (dout_i . v_j).
 *   workspace: device buffer of at least pi_attn_bwd_workspace_size() bytes,
 *   owned by the caller, contents ignored on entry.  Deterministic.
 */
int pi_attn_bwd(const void *q, const void *k, const void *v, const float *alpha,
                const void *out, const float *lse, const void *dout,
                int B, int H, int Hkv, int N, int d, int k_local, int period, int S, int mode,
                void *dq, void *dk, void *dv, float *dalpha,
                void *workspace, size_t workspace_bytes, void *stream);

/* pi_attn_bwd_f32 -- same with fp32 tensors. */
int pi_attn_bwd_f32(const void *q, const void *k, const void *v, const float *alpha,
                    const void *out, const float *lse, const void *dout,
                    int B, int H, int Hkv, int N, int d, int k_local, int period, int S,
                    int mode, void *dq, void *dk, void *dv, float *dalpha,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * pi_attn_fwd_shard -- pi_attn_fwd for one shard of a sequence split over
 * devices (the "pi-Attention" page, section 2, item 2: the periodic skips suit
 * collective communication; its efficiency results are on 8 GPUs).  A shard owns
 * the queries at global positions [t0, t0 + Nq); it holds, in local buffers, the
 * key/value rows of a window [w0, w0 + Nkv) of the sequence that contains every
 * key those queries attend (its own rows and a halo received from other shards;
 * window rows that no query attends may hold anything finite, e.g. zeros).
 * q_offset = t0 - w0 is the key row of the shard's first query.
 *   q, out [B,H,Nq,d] and alpha, lse [B,H,Nq] (the shard's queries); k, v
 *   [B,Hkv,Nkv,d] (the window).  Row r of q is the query at key row q_offset + r;
 *   inside the window every rule of pi_attn_fwd holds with positions taken
 *   relative to w0, so the window must start where the neighbour sets do not
 *   change under the shift: w0 = 0, or every key of every shard query inside the
 *   window (the skips i - m*period and the band), and in ECP mode w0 a multiple
 *   of c = k_local.  The result is then identical to rows [t0, t0 + Nq) of
 *   pi_attn_fwd over the whole sequence.
 *   Requirements: 0 <= q_offset, q_offset + Nq <= Nkv, q_offset a multiple of
 *   128 (else PI_ERR_SHAPE).  bf16; other arguments, errors and rules as
 *   pi_attn_fwd (N there is Nkv here).
 */
int pi_attn_fwd_shard(const void *q, const void *k, const void *v, const float *alpha,
                      int B, int H, int Hkv, int Nq, int Nkv, int q_offset, int d, int k_local,
                      int period, int S, int mode, void *out, float *lse, void *stream);

/*
 * pi_attn_bwd_shard -- pi_attn_bwd for the shard of pi_attn_fwd_shard.
 *   q, out, dout, dq [B,H,Nq,d], alpha, lse, dalpha [B,H,Nq] (the shard's
 *   queries); k, v, dk, dv [B,Hkv,Nkv,d] (the window).  dq and dalpha are the
 *   shard's rows of the whole-sequence gradients.  dk and dv are this shard's
 *   queries' part of the gradients of the window's rows: the whole-sequence dk
 *   and dv of a key row are the sum of these parts over every shard whose window
 *   holds it (the halo rows' parts go back to the shards that own them).
 *   workspace: at least pi_attn_bwd_workspace_size(B, H, Hkv, Nq, d) bytes.
 *   Window requirements as pi_attn_fwd_shard; other rules as pi_attn_bwd.
 */
int pi_attn_bwd_shard(const void *q, const void *k, const void *v, const float *alpha,
                      const void *out, const float *lse, const void *dout,
                      int B, int H, int Hkv, int Nq, int Nkv, int q_offset, int d, int k_local,
                      int period, int S, int mode, void *dq, void *dk, void *dv, float *dalpha,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * pi_attn_bwd_noalloc -- the bf16 backward of pi_attn_bwd, for callers that
 * cannot hand the library a workspace and must not allocate device memory
 * themselves.  The paper has no counterpart to this entry point; it exists
 * for deployment.  Examples of such callers: a serving runtime that reserved
 * the device memory up front for its own pool, where a cudaMalloc would fail
 * or fragment that reservation; code on a latency-critical path, where
 * cudaFree's implicit device-wide synchronisation is not acceptable; and
 * language bindings that only forward the buffers they were given.
 *
 * Arguments, layouts and results are those of pi_attn_bwd without the
 * workspace.  The scratch memory (one fp32 per query row) is a fixed
 * file-scope device array of PI_ATTN_NOALLOC_MAX_ROWS floats (4 MiB), which
 * every GPU that loads the library holds until the process exits.
 *   - B*H*N above PI_ATTN_NOALLOC_MAX_ROWS returns PI_ERR_WORKSPACE and
 *     launches nothing.
 *   - The first call on each device looks up that device's address of the
 *     array (cudaGetSymbolAddress, with the device current) and caches it;
 *     make that first call before any stream capture.  It never calls
 *     cudaMalloc, cudaFree or any allocating routine.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     Nothing in it has to start at zero: each call writes every entry it
 *     reads.  Calls whose kernels overlap on the GPU (different streams
 *     without ordering between them) race on the array and give undefined
 *     results; order them on one stream or with events.
 *   - The cached address belongs to the device's current context: after
 *     cudaDeviceReset on a device, make no further call of this library on it
 *     in the same process (the same holds for the status word of every entry
 *     point).
 */
#define PI_ATTN_NOALLOC_MAX_ROWS (1 << 20)
int pi_attn_bwd_noalloc(const void *q, const void *k, const void *v, const float *alpha,
                        const void *out, const float *lse, const void *dout,
                        int B, int H, int Hkv, int N, int d, int k_local, int period, int S,
                        int mode, void *dq, void *dk, void *dv, float *dalpha, void *stream);

/*
 * pi_attn_decode -- one decode step against a KV cache: for every batch entry b
 * and query head h, row i = N - 1 of pi_attn_fwd, where the cache already holds
 * the key and value rows 0 .. N-1 (the new token's own row at N - 1).  Causal pi
 * mode or ECP mode (bidirectional: PI_ERR_UNSUPPORTED; the future does not exist
 * yet).  The neighbour set of row N-1 is the band rows max(0, N-1-k_local) .. N-1
 * (ECP: the half-segments of row N-1) and the skip rows N-1 - m*period with
 * m*period > k_local, so only those rows of the cache are read.
 *   q [B,H,d] bf16 (the new queries), k_cache and v_cache [B,Hkv,N,d] bf16 (the
 *   layout of pi_attn_fwd's k and v), alpha [B,H] fp32 (the new token's gate;
 *   NULL in ECP mode), out [B,H,d] bf16, lse [B,H] fp32.  d in {64, 128};
 *   H / Hkv <= 16.  Same ownership, asynchrony and error rules as pi_attn_fwd.
 */
int pi_attn_decode(const void *q, const void *k_cache, const void *v_cache, const float *alpha,
                   int B, int H, int Hkv, int N, int d, int k_local, int period, int S, int mode,
                   void *out, float *lse, void *stream);

/*
 * pi_attn_status -- synchronises `stream`, reads the current device's status
 * word, resets it to PI_OK and returns what it held (PI_OK or
 * PI_ERR_DEVICE_TIMEOUT), or PI_ERR_CUDA if the synchronisation failed.
 */
int pi_attn_status(void *stream);

/* pi_attn_strerror -- static, human-readable name of a pi_status_t. */
const char *pi_attn_strerror(int code);

/*
 * pi_attn_debug_counts -- runs the forward (dtype 0 = bf16 kernel chosen as in
 * pi_attn_fwd, 1 = fp32 kernel) and, from that kernel's own tile walk and
 * masks, also writes count [B,H,N] int32 = number of keys the row attended
 * and idx_sum [B,H,N] int64 = sum of their key positions.  Used to check the
 * neighbour enumeration bit-exactly.  Arguments otherwise as pi_attn_fwd.
 */
int pi_attn_debug_counts(const void *q, const void *k, const void *v, const float *alpha,
                         int B, int H, int Hkv, int N, int d, int k_local, int period, int S,
                         int mode, int dtype, void *out, float *lse, int *count,
                         long long *idx_sum, void *stream);

/*
 * pi_attn_debug_probs -- for N <= 2048: runs the forward (writing out and lse
 * as pi_attn_fwd does) and, from the same kernel's tile walk and masks, writes
 * the normalised probability exp(z_ij - lse_in_i) into P [B,H,N,N] fp32 for
 * every key j the row attends to; lse_in must be the lse of an earlier forward
 * on the same inputs.  Entries for keys the row does not attend to are not
 * written: the caller zero-fills P.  dtype as in pi_attn_debug_counts.
 */
int pi_attn_debug_probs(const void *q, const void *k, const void *v, const float *alpha,
                        const float *lse_in, int B, int H, int Hkv, int N, int d, int k_local,
                        int period, int S, int mode, int dtype, void *out, float *lse, float *P,
                        void *stream);

/*
 * pi_attn_debug_trace -- runs the bf16 tcgen05 forward (d = 64 or 128; writes out
 * and lse as pi_attn_fwd does) and records, for CTAs 0 .. n_trace_ctas-1, the
 * SM cycle counter (clock64) at the pipeline events of each CTA into
 * trace [n_trace_ctas][240] int64 (caller-owned, zero-filled by the caller):
 *   slot 0 entry, 1 set-up done, 2 Q load issued, 3 Q landed (seen by the S
 *   issuer), 4 O complete (seen by the epilogue), 5 output stored, 6 exit,
 *   7 number of key tiles; for tile t < 16: 8+t K load issued, 24+t V load
 *   issued, 40+t S = QK^T issued, 56+t O += PV issued, 72+t S seen by the
 *   softmax, 88+t P ready; and cycles spent in waits, each measured within
 *   one thread: 104+t S issuer waiting for K, 120+t S issuer waiting for its
 *   TMEM buffer, 136+t PV issuer waiting for P, 152+t PV issuer waiting for V,
 *   168+t softmax waiting for S; softmax stamps inside tile t: 184+t S loaded
 *   from TMEM, 200+t maxima done, 216+t P stored to TMEM; 232 the SM id, 233
 *   and 234 the global timer (ns) at entry and exit.  Stamps of different warps
 *   need not share a clock.  A profiling aid; the pages define no such
 *   operation.
 */
int pi_attn_debug_trace(const void *q, const void *k, const void *v, const float *alpha,
                        int B, int H, int Hkv, int N, int d, int k_local, int period, int S,
                        int mode, void *out, float *lse, long long *trace, int n_trace_ctas,
                        void *stream);

/*
 * pi_attn_debug_wait_timeout -- launches one block that waits on a shared-memory
 * barrier nothing ever completes, giving up after timeout_us microseconds;
 * it then records PI_ERR_DEVICE_TIMEOUT in the status word and returns.
 * Exercises the bounded-wait error path without faulting the GPU.
 */
int pi_attn_debug_wait_timeout(int timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PI_ATTN_H_ */
