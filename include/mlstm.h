/*
 * mlstm.h - C ABI of libmlstm.so, the GB300 (sm_103a) mLSTM matrix-memory path.
 *
 * Method: "xLSTM: Extended Long Short-Term Memory".
 *   part 28/30 "Parallel mLSTM Forward Pass", eqs (71)-(77), and its stabilized
 *   summary eqs (79)-(86) with the log forget matrix eq (101);
 *   the recurrent mLSTM whose backward pass is eqs (59)-(70) (part 28/30),
 *   with the output gate eq (27) (part 17/30) for generation.
 *
 * Conventions shared by every entry point
 *  - All tensors are dense, row-major, last index fastest, in DEVICE memory
 *    owned by the caller.  The library never allocates, frees or retains them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls only enqueue work on it; they do not synchronize.
 *  - Every call returns an mlstm_status.  Argument errors are detected on the
 *    host before anything is launched and leave all buffers untouched.  Calls
 *    never abort the process.
 *  - The kernels' internal waits are bounded.  A wait that runs out sets a
 *    device-side status word and the kernel returns early (its outputs are then
 *    undefined); mlstm_last_device_status() reads and clears that word.
 *  - k enters scaled by 1/sqrt(d_qk) (the factor is moved onto K below eq 76);
 *    q is not scaled.  Both entry points take the raw k.
 *  - dtype: MLSTM_F32 or MLSTM_BF16 for q, k, v, o and the output h.  Gate
 *    pre-activations, the stabilizer m, the normalizer n and the state (C, n,
 *    m) are always fp32.  Arithmetic is fp32 (bf16 tensor-core products with
 *    fp32 accumulation on the bf16 path).
 */
#ifndef MLSTM_H
#define MLSTM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLSTM_OK = 0,
    MLSTM_EINVAL = -1,       /* a size, pointer or combination is invalid */
    MLSTM_EALIGN = -2,       /* a pointer is not 16-byte aligned */
    MLSTM_EDTYPE = -3,       /* unsupported dtype */
    MLSTM_ECUDA = -4,        /* a CUDA runtime/driver call failed */
    MLSTM_ETIMEOUT = -5,     /* a kernel's bounded wait ran out (device status) */
    MLSTM_EUNSUPPORTED = -6, /* valid arguments this build or device cannot run */
    MLSTM_EWORKSPACE = -7    /* workspace missing or smaller than required */
} mlstm_status;

typedef enum { MLSTM_F32 = 0, MLSTM_BF16 = 1 } mlstm_dtype;

/* Kernel choice for mlstm_parallel_fwd_ex. */
typedef enum {
    MLSTM_ALGO_AUTO = 0, /* tensor-core kernel when the shape allows, else SIMT */
    MLSTM_ALGO_SIMT = 1, /* fp32 CUDA-core kernel: any d_qk, d_v <= 512 (fp32 or bf16) */
    MLSTM_ALGO_TC = 2    /* tcgen05/TMEM kernel: bf16, d_qk and d_v multiples of 64, <= 512 */
} mlstm_algo;

/* Bytes of device workspace mlstm_parallel_fwd needs for B*H sequences of
 * length T: the per-token gate terms of eqs (79)-(80) and (101), 3 fp32 per
 * token, rounded up to 256 bytes.  Returns 0 if any size is negative. */
size_t mlstm_parallel_fwd_workspace(int B, int H, int T);

/* Stabilized parallel mLSTM forward pass, part 28/30 eqs (79)-(86):
 *   Fbar_ij = sum_{k=j+1..i} log sigmoid(fgate_pre_k)    (eq 101, j <= i)
 *   D~_ij   = Fbar_ij + igate_pre_j,  m_i = max_{j<=i} D~_ij        (79)-(80)
 *   C'_ij   = (q_i . k_j)/sqrt(d_qk) * exp(D~_ij - m_i)              (81)-(82)
 *   b_i = sum_j C'_ij,  n_i = max(|b_i|, exp(-m_i))                   (83)-(84)
 *   h_i = sum_j (C'_ij / n_i) v_j                                     (85)-(86)
 * (H~ of eq 77; the output gate of eq 78 is not applied.)
 *
 *   q, k       [B,H,T,d_qk]  dtype
 *   v          [B,H,T,d_v]   dtype
 *   igate_pre  [B,H,T] fp32   input-gate pre-activations i~
 *   fgate_pre  [B,H,T] fp32   forget-gate pre-activations f~
 *   h          [B,H,T,d_v]   dtype, output
 *   m_out      [B,H,T] fp32   output, may be NULL: row stabilizer m_i
 *   n_out      [B,H,T] fp32   output, may be NULL: normalizer n_i
 *   workspace  >= mlstm_parallel_fwd_workspace(B,H,T) bytes of device memory,
 *              16-byte aligned; contents on entry are ignored.
 * Requirements: B,H >= 0, T >= 0, 1 <= d_qk, d_v <= 512, d_qk and d_v
 * multiples of 8 (fp32: multiples of 4); q, k, v, h 16-byte aligned.
 * B*H*T == 0 is a no-op returning MLSTM_OK.  If a row's n_i is 0 (all its
 * C'_ij are exactly 0 and exp(-m_i) underflows), its h_i is written as 0. */
int mlstm_parallel_fwd(const void *q, const void *k, const void *v,
                       const float *igate_pre, const float *fgate_pre,
                       void *h, float *m_out, float *n_out,
                       int B, int H, int T, int d_qk, int d_v, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream);

/* mlstm_parallel_fwd with an explicit kernel choice (mlstm_algo).  Returns
 * MLSTM_EUNSUPPORTED if the forced kernel cannot run this shape or dtype. */
int mlstm_parallel_fwd_ex(const void *q, const void *k, const void *v,
                          const float *igate_pre, const float *fgate_pre,
                          void *h, float *m_out, float *n_out,
                          int B, int H, int T, int d_qk, int d_v, int dtype,
                          void *workspace, size_t workspace_bytes, int algo, void *stream);

/* The two phases of mlstm_parallel_fwd_ex, for callers that time or reuse
 * them separately.
 *
 * mlstm_gate_prep: the gate terms of eqs (79)-(81) and (101) for every token,
 * written to `workspace` (>= mlstm_parallel_fwd_workspace(B,H,T) bytes):
 *   cs_t = sum_{k<=t} log sigmoid(fgate_pre_k)     (fp32 two-sum accumulation)
 *   a_t  = igate_pre_t - cs_t,  m_t = cs_t + max_{j<=t} a_j   (row max, eq 80)
 * stored as three fp32 arrays of B*H*T entries, each starting on a 256-byte
 * boundary: a_t*log2(e), max_{j<=t} a_j*log2(e), m_t.
 *
 * mlstm_parallel_fwd_gated: eqs (81)-(86) from those terms; same arguments and
 * rules as mlstm_parallel_fwd_ex minus the gate pre-activations.  The
 * workspace must hold the output of mlstm_gate_prep for the same B, H, T. */
int mlstm_gate_prep(const float *igate_pre, const float *fgate_pre, int B, int H, int T,
                    void *workspace, size_t workspace_bytes, void *stream);

int mlstm_parallel_fwd_gated(const void *q, const void *k, const void *v,
                             void *h, float *m_out, float *n_out,
                             int B, int H, int T, int d_qk, int d_v, int dtype,
                             const void *workspace, size_t workspace_bytes, int algo,
                             void *stream);

/* The recurrent state after the last token of each sequence, from the gate
 * terms of the parallel pass: the hand-off from a parallel prefill to
 * mlstm_step / mlstm_step_seq.  Unrolling the stabilized recurrence (part
 * 28/30 eqs 59-70) from C = 0, n = 0, m = -inf over t = 1..T gives
 *   m = m_T (the last row's max of eq 80),
 *   C = sum_j D'_Tj v_j (k_j/sqrt(d_qk))^T,   n = sum_j D'_Tj k_j/sqrt(d_qk),
 * where D'_Tj = exp(D~_Tj - m_T) is the last row of the stabilized gate
 * matrix of eq (81); (C, n) are stored times exp(-m) as mlstm_step expects.
 *
 *   k          [B,H,T,d_qk] dtype,  v [B,H,T,d_v] dtype (the same as passed
 *              to the parallel forward)
 *   workspace  the gate terms of the same B, H, T, as left by
 *              mlstm_gate_prep, mlstm_parallel_fwd or mlstm_parallel_fwd_ex
 *   C          [B,H,d_v,d_qk] fp32 out,  n [B,H,d_qk] fp32 out,  m [B,H] fp32 out
 * Requirements as for mlstm_parallel_fwd_gated (T >= 1), and C, n 16-byte
 * aligned.  The outputs are overwritten; they may not alias k, v or the
 * workspace. */
int mlstm_parallel_final_state(const void *k, const void *v, const void *workspace, size_t workspace_bytes,
                               float *C, float *n, float *m, int B, int H, int T, int d_qk, int d_v,
                               int dtype, void *stream);

/* mlstm_parallel_fwd on inputs and an output in host memory: the call a
 * caller makes whose tensors live on the CPU side.  The heads are processed
 * in up to 8 chunks; each chunk's upload, its forward pass and its download
 * overlap with those of its neighbours (two library-owned copy streams plus
 * `stream` for the compute, two device buffers per operand in `workspace`).
 * Results are identical to mlstm_parallel_fwd on the same data.
 *
 *   q, k, v, igate_pre, fgate_pre, h   as in mlstm_parallel_fwd, but host
 *              pointers.  Page-locked memory (cudaHostAlloc, cudaHostRegister)
 *              lets the copies run asynchronously and overlap; pageable
 *              memory is correct but serialises them.
 *   workspace  device memory of mlstm_parallel_fwd_host_workspace(...) bytes,
 *              256-byte aligned, owned by the caller; no two calls that may
 *              run at the same time may share it.
 * The call returns once everything is queued; `stream` completes when h is
 * in host memory (synchronise `stream` before reading h).  The library's copy
 * streams and events are created on the first call on each device and kept;
 * calls from several host threads are serialised while they queue work. */
size_t mlstm_parallel_fwd_host_workspace(int B, int H, int T, int d_qk, int d_v, int dtype);

int mlstm_parallel_fwd_host(const void *q, const void *k, const void *v,
                            const float *igate_pre, const float *fgate_pre, void *h,
                            int B, int H, int T, int d_qk, int d_v, int dtype,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Options of the *_opt entry points; a zero-initialised struct (or a NULL
 * pointer) gives the behaviour of the plain entry points.
 *   algo        MLSTM_ALGO_* (the parallel forward; ignored elsewhere)
 *   forget_exp  0: forget gate f = sigmoid(f~), log f = log sigmoid(f~) (the
 *               form the parallel equations fix, part 28/30 eqs 71, 101);
 *               1: f = exp(f~), log f = f~ (part 28/30 eq 70: the activation
 *               may be sigma or exp).
 *   ogate_pre   the parallel forward only: [B,H,T,d_v] dtype output-gate
 *               pre-activations, 16-byte aligned, or NULL.  When given, h =
 *               sigmoid(ogate_pre) (.) H~ (eq 78) instead of H~ (eq 77); the
 *               CTA-pair kernel applies it in its epilogue, the other kernels
 *               in a separate elementwise pass.
 *   b_out       the parallel forward only: [B,H,T] fp32 out, the signed row
 *               sums b of eq (83) (n = max(|b|, exp(-m))), or NULL.  With H~
 *               and n they are what mlstm_parallel_bwd_saved takes. */
typedef struct {
    int algo;
    int forget_exp;
    const void *ogate_pre;
    float *b_out;
} mlstm_options;

int mlstm_parallel_fwd_opt(const void *q, const void *k, const void *v,
                           const float *igate_pre, const float *fgate_pre,
                           void *h, float *m_out, float *n_out,
                           int B, int H, int T, int d_qk, int d_v, int dtype,
                           void *workspace, size_t workspace_bytes,
                           const mlstm_options *opt, void *stream);

/* mlstm_gate_prep with options (forget_exp); the gate terms then serve
 * mlstm_parallel_fwd_gated and mlstm_parallel_final_state as usual. */
int mlstm_gate_prep_opt(const float *igate_pre, const float *fgate_pre, int B, int H, int T,
                        void *workspace, size_t workspace_bytes, const mlstm_options *opt,
                        void *stream);

/* mlstm_step_seq with options (forget_exp); L = 1 is one mlstm_step. */
int mlstm_step_seq_opt(float *C, float *n, float *m,
                       const void *q, const void *k, const void *v, const void *o,
                       const float *igate_pre, const float *fgate_pre, void *h,
                       int B, int H, int L, int d_qk, int d_v, int dtype,
                       const mlstm_options *opt, void *stream);

/* Backward pass of mlstm_parallel_fwd (part 28/30 eqs 87-105): given the
 * output gradient dh = dL/dH~, the gradients of q, k, v and of the gate
 * pre-activations.  The stabilizer m is held constant, as on the pages (its
 * gradients cancel); eq (90) is read with sign(b), the derivative of |b|.
 * (mlstm_parallel_bwd_opt below adds the output gate and the exponential
 * forget activation.)
 *
 *   q, k, v, igate_pre, fgate_pre   the forward's inputs (layouts as there)
 *   dh         [B,H,T,d_v]  dtype: dL/dH~
 *   dq, dk     [B,H,T,d_qk] dtype out,   dv [B,H,T,d_v] dtype out
 *   d_igate, d_fgate  [B,H,T] fp32 out
 *   workspace  256-byte aligned device memory of
 *              mlstm_parallel_bwd_workspace_ex(B,H,T,d_qk,d_v,dtype) bytes
 *              (the size of the path that will run), or of
 *              mlstm_parallel_bwd_workspace(B,H,T,dtype) bytes (enough for
 *              either path).
 * Two paths:
 *  - bf16 with d_qk and d_v multiples of 8, on the sm_100 family: a forward
 *    pass gives H~, n and the signed row sums b; a persistent tensor-core
 *    kernel forms S = QK^T/sqrt(d) and dC = dH~ V^T per 128 x 128 tile on or
 *    below the diagonal in TMEM and writes G = D' (.) dC~' and P = C~'/n
 *    (bf16) and the tile's row and column sums of dD~; a second tensor-core
 *    kernel forms dQ, dK, dV over the lower triangle of G and P.  Workspace:
 *    two bf16 T x T matrices per head (about 0.54 GB for B=8, H=4, T=2048).
 *  - otherwise (fp32, or shapes the tensor-core kernels do not tile) the five
 *    T x T products run in a batched CUDA-core GEMM kernel of the library
 *    (fp32 accumulation, each over its causal part only), with fp32 S and
 *    dL/dC materialised (about 1.6 GB for B=8, H=4, T=2048, bf16).
 * Requirements: 1 <= T <= 16384; 1 <= d_qk, d_v <= 512; no output may alias
 * an input. */
size_t mlstm_parallel_bwd_workspace(int B, int H, int T, int dtype);
size_t mlstm_parallel_bwd_workspace_ex(int B, int H, int T, int d_qk, int d_v, int dtype);

/* mlstm_parallel_bwd given what the forward already produced, as a training
 * step keeps it: h = H~ (the forward's output without an output gate), n
 * (its n_out) and b (its options' b_out), all from mlstm_parallel_fwd_opt
 * on the same inputs.  On the tensor-core path the forward pass inside the
 * backward is then skipped; otherwise h, n, b are ignored and the result is
 * that of mlstm_parallel_bwd.  Arguments and workspace as there, plus
 *   h          [B,H,T,d_v] dtype, n, b [B,H,T] fp32 (all non-NULL). */
int mlstm_parallel_bwd_saved(const void *q, const void *k, const void *v,
                             const float *igate_pre, const float *fgate_pre, const void *dh,
                             const void *h, const float *n, const float *b,
                             void *dq, void *dk, void *dv, float *d_igate, float *d_fgate,
                             int B, int H, int T, int d_qk, int d_v, int dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

int mlstm_parallel_bwd(const void *q, const void *k, const void *v,
                       const float *igate_pre, const float *fgate_pre, const void *dh,
                       void *dq, void *dk, void *dv, float *d_igate, float *d_fgate,
                       int B, int H, int T, int d_qk, int d_v, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream);

/* mlstm_parallel_bwd with options: the backward of mlstm_parallel_fwd_opt.
 *   opt->forget_exp  the exponential forget activation (log f = f~, part
 *               28/30 eq 70's gamma = exp): d f~ = dL/dlog f instead of
 *               sigmoid(-f~) dL/dlog f (eq 104)
 *   opt->ogate_pre   [B,H,T,d_v] dtype output-gate pre-activations, or NULL.
 *               When given, the forward was h = sigmoid(o~) (.) H~ (eq 78),
 *               dh is dL/dh, and d_ogate ([B,H,T,d_v] dtype out, required)
 *               receives dL/do~ = dh (.) H~ (.) sigmoid(o~)(1 - sigmoid(o~));
 *               the rest of the backward runs on dL/dH~ = dh (.) sigmoid(o~).
 *   opt->algo, opt->b_out are ignored.
 *   h_saved, n_saved, b_saved   all NULL, or all given as for
 *               mlstm_parallel_bwd_saved: H~ (the forward's output WITHOUT the
 *               output gate, i.e. of mlstm_parallel_fwd_opt with ogate_pre
 *               NULL), n and the signed b of the forward on the same inputs
 *               and forget activation.
 *   workspace   mlstm_parallel_bwd_workspace_opt(B,H,T,d_qk,d_v,dtype,opt)
 *               bytes (256-byte aligned): the path's workspace, plus one
 *               [B,H,T,d_v] dtype buffer with an output gate (two on the
 *               CUDA-core path, which also forms H~).
 * Other arguments, requirements and errors as mlstm_parallel_bwd;
 * MLSTM_EINVAL when only some of h_saved, n_saved, b_saved are given or
 * ogate_pre is set without d_ogate. */
size_t mlstm_parallel_bwd_workspace_opt(int B, int H, int T, int d_qk, int d_v, int dtype,
                                        const mlstm_options *opt);

int mlstm_parallel_bwd_opt(const void *q, const void *k, const void *v,
                           const float *igate_pre, const float *fgate_pre, const void *dh,
                           const void *h_saved, const float *n_saved, const float *b_saved,
                           void *dq, void *dk, void *dv, float *d_igate, float *d_fgate, void *d_ogate,
                           int B, int H, int T, int d_qk, int d_v, int dtype,
                           void *workspace, size_t workspace_bytes,
                           const mlstm_options *opt, void *stream);

/* Backward pass of the recurrent form (backpropagation through time, part
 * 28/30 eqs 59-70) of the cell the recurrent step and mlstm_step_seq compute
 * from a fresh state, for the output gradient dh = dL/dh:
 *   C_t = f_t C_{t-1} + i_t v_t (s k_t)^T,  n_t = f_t n_{t-1} + i_t s k_t,
 *   h_t = sigmoid(o~_t) (.) C_t q_t / max(|n_t . q_t|, 1),
 * i_t = exp(i~_t), f_t = sigmoid(f~_t) (exp(f~_t) with forget_exp),
 * s = 1/sqrt(d_qk), C_{-1} = 0, n_{-1} = 0.  Evaluated with the stabilized
 * states (the result is that of the unstabilized recurrence); the gradient of
 * the forget pre-activation uses the exact identity dL/dlog f_t =
 * sum_{u>=t} (q_u . dq_u - k_u . dk_u), equal to eq (68).
 *
 *   q, k       [B,H,T,d_qk] dtype, 16-byte aligned;  v [B,H,T,d_v] dtype
 *   igate_pre, fgate_pre   [B,H,T] fp32
 *   dh         [B,H,T,d_v] dtype: dL/dh (dL/dH~ without an output gate)
 *   dq, dk     [B,H,T,d_qk] dtype out,  dv [B,H,T,d_v] dtype out
 *   d_igate, d_fgate       [B,H,T] fp32 out
 *   d_ogate    [B,H,T,d_v] dtype out, required when opt->ogate_pre is set
 *              (eq 70), else ignored
 *   opt        NULL or: forget_exp (exponential forget activation) and
 *              ogate_pre ([B,H,T,d_v] dtype output-gate pre-activations, or
 *              NULL); algo is ignored
 *   workspace  mlstm_recurrent_bwd_workspace(B,H,T,d_qk,d_v) bytes of device
 *              memory, 256-byte aligned: per-CTA shares of dq and dk
 *              (2 ceil(d_v/64) fp32 rows of d_qk per token) and three fp32
 *              values per token, so it grows as B*H*T (about 1.2 GB for B=8,
 *              H=4, T=2048, d=384).
 * Requirements: 1 <= d_qk, d_v <= 512, d_qk a multiple of 8; no output may
 * alias an input.  B*H*T = 0 returns MLSTM_OK without work.  Four kernels on
 * `stream`: the forward and backward sweeps (state in registers, 64 or 96
 * rows of one head per CTA: 96 when those CTAs fill the GPU in one wave), the
 * per-token combination, the per-head suffix sums. */
size_t mlstm_recurrent_bwd_workspace(int B, int H, int T, int d_qk, int d_v);

int mlstm_recurrent_bwd(const void *q, const void *k, const void *v,
                        const float *igate_pre, const float *fgate_pre, const void *dh,
                        void *dq, void *dk, void *dv, float *d_igate, float *d_fgate, void *d_ogate,
                        int B, int H, int T, int d_qk, int d_v, int dtype,
                        void *workspace, size_t workspace_bytes,
                        const mlstm_options *opt, void *stream);

/* One stabilized recurrent mLSTM step for every head, the generation step
 * (the recurrence differentiated by part 28/30 eqs 59-70, output gate eq 27):
 *   m'  = max(log sigmoid(f~) + m, i~)
 *   f'  = exp(log sigmoid(f~) + m - m'),   i' = exp(i~ - m')
 *   C  <- f' C + i' v (k/sqrt(d_qk))^T,    n <- f' n + i' k/sqrt(d_qk)
 *   h   = sigmoid(o) * (C q) / max(|n . q|, exp(-m'))
 * The stored (C, n) is the true state times exp(-m).  A fresh sequence starts
 * from C = 0, n = 0, m = -inf.
 *
 *   C          [B,H,d_v,d_qk] fp32  in/out (updated in place)
 *   n          [B,H,d_qk]     fp32  in/out
 *   m          [B,H]          fp32  in/out
 *   q, k       [B,H,d_qk]     dtype
 *   v          [B,H,d_v]      dtype
 *   o          [B,H,d_v]      dtype output-gate pre-activations, or NULL for
 *                             no output gate (h = h~)
 *   igate_pre, fgate_pre [B,H] fp32
 *   h          [B,H,d_v]      dtype output
 * Requirements: B,H >= 0; 1 <= d_qk, d_v <= 512; d_qk a multiple of 8;
 * C, n, q, k 16-byte aligned.  h may not alias any input. */
int mlstm_step(float *C, float *n, float *m,
               const void *q, const void *k, const void *v, const void *o,
               const float *igate_pre, const float *fgate_pre, void *h,
               int B, int H, int d_qk, int d_v, int dtype, void *stream);

/* L consecutive recurrent steps for every head in one call: recurrent
 * prefill of a prompt, or several generated tokens at once.  The result is
 * exactly that of mlstm_step applied for t = 0, 1, ..., L-1 in order (same
 * recurrence, same state convention, same output gate), but the state is
 * read from and written to memory once instead of L times: each head's C
 * stays on chip for the whole run.
 *
 *   C, n, m    as in mlstm_step: the state before token 0 on entry, the state
 *              after token L-1 on return (updated in place)
 *   q, k       [B,H,L,d_qk]  dtype
 *   v          [B,H,L,d_v]   dtype
 *   o          [B,H,L,d_v]   dtype, or NULL for no output gate
 *   igate_pre, fgate_pre [B,H,L] fp32
 *   h          [B,H,L,d_v]   dtype output, token t of head (b,h) at
 *              ((b*H + h)*L + t)*d_v
 * Requirements: B,H,L >= 0; 1 <= d_qk, d_v <= 512; d_qk a multiple of 8;
 * C, n, q, k 16-byte aligned.  h may not alias any input.  L = 0 leaves the
 * state unchanged and launches nothing. */
int mlstm_step_seq(float *C, float *n, float *m,
                   const void *q, const void *k, const void *v, const void *o,
                   const float *igate_pre, const float *fgate_pre, void *h,
                   int B, int H, int L, int d_qk, int d_v, int dtype, void *stream);

/* Size of the scratch array built into the library for
 * mlstm_parallel_fwd_noalloc: 4 MiB, enough for B*H*T up to 349,504 tokens. */
#define MLSTM_NOALLOC_SCRATCH_BYTES (4u << 20)

/* mlstm_parallel_fwd for callers that cannot allocate device memory.  (The
 * paper has no counterpart to this entry point; it is a library convenience.)
 *
 * Who needs it: code that must not call cudaMalloc or any allocating routine,
 * for example a plug-in whose host application owns all device memory, a
 * caller working inside a memory pool's own callbacks, or a job whose memory
 * budget is fixed up front.  Such callers cannot provide the workspace that
 * mlstm_parallel_fwd asks for.  This entry point instead uses a fixed scratch
 * array of MLSTM_NOALLOC_SCRATCH_BYTES compiled into the library.  Every GPU
 * that loads the library holds that array until the process exits.
 *
 * Same arguments, results and rules as mlstm_parallel_fwd, minus the
 * workspace; the caller still passes all inputs and outputs.  It allocates
 * nothing.
 *  - Returns MLSTM_EWORKSPACE, and launches nothing, when the job needs more
 *    scratch than the array holds: mlstm_parallel_fwd_workspace(B,H,T) >
 *    MLSTM_NOALLOC_SCRATCH_BYTES.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call before any stream capture begins.
 *  - Every call on a device shares the one array.  Calls whose kernels
 *    overlap on the GPU (other streams, other host threads) race on it and
 *    give wrong results: serialize them.  Nothing in the array needs clearing
 *    between calls; each call overwrites what it reads. */
int mlstm_parallel_fwd_noalloc(const void *q, const void *k, const void *v,
                               const float *igate_pre, const float *fgate_pre,
                               void *h, float *m_out, float *n_out,
                               int B, int H, int T, int d_qk, int d_v, int dtype,
                               void *stream);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: MLSTM_OK, or MLSTM_ETIMEOUT if a kernel's bounded wait
 * ran out since the last call.  MLSTM_ECUDA if the synchronization failed. */
int mlstm_last_device_status(void *stream);

/* Spin budget of each bounded wait inside the kernels (iterations of a
 * polling loop).  0 restores the default.  Returns the previous budget.
 * Small budgets make waits give up early; used to test the timeout path. */
long long mlstm_set_spin_limit(long long limit);

/* Static, human-readable name of a status code. */
const char *mlstm_status_str(int status);

/* Library ABI version (major*100 + minor). */
int mlstm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLSTM_H */
