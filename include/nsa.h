/*
 * nsa.h -- C ABI of libnsa.so: Native-Sparse-Attention block-selection
 * attention (forward producing O and LSE, backward producing dQ, dK, dV)
 * under grouped-query attention, on one NVIDIA GB300 (sm_103a).
 *
 * Where the operation is defined.  The gradcheck-gate page
 * ("test_kernel_backward.py", functions run_one and main) fixes the
 * operation: q [B,Hq,T,D], k and v [B,Hkv,T,D], a per-token block index
 * idx = make_block_idx(B, Hkv, T, block_size, S), o = selection forward of
 * (q, k, v, idx, block_size), and dQ, dK, dV = the gradient of <dO, o>.
 * The cuDNN-frontend pull-request page ("port the SM80 backward onto
 * SdpaBwdDsl ...", its description and the review of the THD path) supplies
 * the dense causal backward, the packed THD variable-length form
 * (cum_seqlen tensors), the do_dot pre-pass, caller-owned workspace with no
 * per-call allocation, and respecting the caller's stream.
 *
 * Definitions (G = Hq/Hkv; query head h reads kv head h/G; every index row
 * is shared by the G query heads of its kv head):
 *   sel(t)   = { idx[b,g,t,s] : s < S, idx != -1 }
 *   key k is attended by row t  iff  k <= t  and  k/block_size in sel(t)
 *   P_tk     = exp(scale*q_t.k_k - LSE_t),  LSE_t = log sum_k exp(scale*q_t.k_k)
 *   O_t      = sum_k P_tk v_k
 *   dS_tk    = P_tk (dO_t.v_k - dO_t.O_t)
 *   dQ_t     = scale sum_k dS_tk k_k
 *   dK_k     = scale sum_{h in group, t} dS_tk q_t,   dV_k = sum_{h, t} P_tk dO_t
 * LSE is the natural-log sum.  A row with no attended key gets O = 0,
 * LSE = -inf and contributes no gradient.
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller, in the
 *    layout named by nsa_problem.layout with the strides the problem
 *    declares (dense when they are 0), 16-byte aligned.  The library
 *    never allocates or frees memory and never synchronises: work is
 *    enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *    A launch that can run beside the ones after it (the other-shapes dQ
 *    of a backward) goes on a helper stream the library keeps per device,
 *    forked from `stream` and joined back to it by events: it starts after
 *    the work enqueued on `stream` before the call and ends before the work
 *    enqueued after it, also inside a CUDA-graph capture of `stream`.
 *  - Shape, dtype and layout errors are returned synchronously before any
 *    launch.  Errors found on the device (a bad index entry, a wait that
 *    timed out) are recorded in the workspace and read back with
 *    nsa_get_error.  After any error the outputs are unspecified.
 *  - `ws` is a caller-provided device workspace of at least the size the
 *    matching *_workspace_size function returns (256-byte aligned).  Its
 *    contents on entry do not matter; it must not be shared by calls that
 *    can run at the same time.
 *  - dtype NSA_DTYPE_BF16: q,k,v,o,dO,dq,dk,dv are bfloat16; NSA_DTYPE_F32:
 *    they are float.  lse is always float; idx and cu_seqlens are int32.
 *    Accumulation is fp32 in both cases; results are rounded once.
 */
#ifndef NSA_H
#define NSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nsa_status {
    NSA_OK = 0,
    NSA_ERR_INVALID_ARG = 1,    /* null pointer, bad shape, misaligned pointer */
    NSA_ERR_UNSUPPORTED = 2,    /* valid problem this build does not handle */
    NSA_ERR_BAD_INDEX = 3,      /* (device) index entry < -1, in the future, or repeated in a row */
    NSA_ERR_DEVICE_TIMEOUT = 4, /* (device) a bounded wait inside a kernel gave up */
    NSA_ERR_CUDA = 5,           /* a CUDA runtime call failed (launch, tensor map) */
    NSA_ERR_WORKSPACE = 6       /* ws is NULL, too small or misaligned */
} nsa_status;

enum { NSA_DTYPE_F32 = 0, NSA_DTYPE_BF16 = 1 };

/*
 * Layouts.  BHTD: q,o,dO,dq [B,Hq,T,D]; k,v,dk,dv [B,Hkv,T,D];
 * idx [B,Hkv,T,S]; lse [B,Hq,T].
 * THD (packed variable length, through the entry points that take
 * cu_seqlens): q,o,dO,dq [total,Hq,D]; k,v,dk,dv [total,Hkv,D]; idx
 * [total,Hkv,S] with sequence-local block ids; lse [total,Hq]; cu_seqlens
 * [B+1] int32 with cu_seqlens[0] = 0 and cu_seqlens[B] = total.  Causality
 * and block numbering restart at every sequence.  Query and key lengths are
 * equal except through nsa_causal_*, which take the keys' own cu_seqlens.
 */
enum { NSA_LAYOUT_BHTD = 0, NSA_LAYOUT_THD = 1 };

typedef struct nsa_problem {
    int32_t B;            /* batch size (BHTD) or number of sequences (THD) */
    int32_t Hq;           /* query heads */
    int32_t Hkv;          /* key/value heads; Hq % Hkv == 0 */
    int32_t T;            /* BHTD: sequence length; THD: upper bound on every sequence length */
    int32_t D;            /* head dimension: 32, 64 or 128 */
    int32_t block_size;   /* keys per selectable block: 16, 32 or 64 */
    int32_t S;            /* slots per index row (ignored by the dense entry points) */
    int32_t dtype;        /* NSA_DTYPE_* */
    int32_t layout;       /* NSA_LAYOUT_*; the varlen entry points require THD, the others BHTD */
    int32_t total_tokens; /* THD: cu_seqlens[B]; ignored for BHTD */
    float scale;          /* softmax scale; <= 0 selects 1/sqrt(D) */
    int32_t reserved;     /* set to 0 */
    /*
     * Declared strides (cuDNN-frontend page: the SM80 port's "declared
     * strides", no pad/gather copies of non-compact operands), in ELEMENTS,
     * of (batch, head, token) for each tensor; the head dimension D is always
     * contiguous.  All three 0 selects the dense layout of `layout` (the
     * shapes listed above), so a zero-initialised struct describes dense
     * tensors.  THD: the batch entry is ignored and the token entry is the
     * step between packed rows.  Every stride in use must be positive, a
     * multiple of 16 bytes (8 bf16 or 4 fp32 elements) and below 2^40 bytes,
     * else the call returns NSA_ERR_INVALID_ARG.  Example: q, k, v sliced
     * out of one packed [B, T, Hq + 2*Hkv, D] tensor have (batch, head, token)
     * strides (T*(Hq+2*Hkv)*D, D, (Hq+2*Hkv)*D).  Outputs must not overlap
     * each other or any input.
     */
    int64_t q_stride[3];   /* q */
    int64_t kv_stride[3];  /* k and v */
    int64_t o_stride[3];   /* o (written by the forward, read by the backward) and dO */
    int64_t dq_stride[3];  /* dq */
    int64_t dkv_stride[3]; /* dk and dv */
    /*
     * Keys with their own lengths -- read by the nsa_causal_* entry points
     * only (every other entry point has keys and queries of equal length):
     *   Tk           BHTD: key length of every sequence; THD: an upper bound
     *                on every key length; 0 means T
     *   total_keys   THD: cu_seqlens_k[B] (at least 1); ignored for BHTD
     *   bottom_right 0: row t of a sequence sits at key position t (the
     *                diagonal of the top-left corner); 1: at t + Lk - Lq
     *                (the bottom-right corner, so the last query row sees
     *                every key)
     */
    int32_t Tk;
    int32_t total_keys;
    int32_t bottom_right;
    int32_t reserved2;     /* set to 0 */
} nsa_problem;

/* Workspace bytes needed by the forward / backward entry points (0 on an invalid problem).
 * nsa_sel_fwd_workspace_size / nsa_sel_bwd_workspace_size are the same functions under
 * the selection entries' names. */
size_t nsa_fwd_workspace_size(const nsa_problem *p);
size_t nsa_bwd_workspace_size(const nsa_problem *p);
size_t nsa_sel_fwd_workspace_size(const nsa_problem *p);
size_t nsa_sel_bwd_workspace_size(const nsa_problem *p);

/*
 * Selection forward (gradcheck-gate page: the selection forward called in
 * run_one with (q, k, v, idx, block_size)).  Writes o (layout of q) and
 * lse.  idx rows may hold -1 anywhere; entries are validated on the device.
 */
nsa_status nsa_sel_fwd(const nsa_problem *p, const void *q, const void *k, const void *v,
                       const int32_t *block_idx, void *o, float *lse, void *ws, size_t ws_bytes,
                       void *stream);

/*
 * Selection backward (gradcheck-gate page: o.backward(dO) through the
 * selection forward; cuDNN-frontend page: the backward chain do_dot ->
 * main -> dQ -> GQA reduction).  Inputs are the forward's inputs plus its
 * o and lse and the upstream gradient dO; writes dq, dk, dv (layouts of q
 * and k).  Runs: D_t = rowsum(dO*O); the block -> token inverse index;
 * dK/dV per (kv block, kv head) summed over the G query heads in-kernel with
 * a fixed summation order (deterministic, no atomics on data); dQ per query
 * tile.  Every output element is written exactly once.
 */
nsa_status nsa_sel_bwd(const nsa_problem *p, const void *q, const void *k, const void *v,
                       const void *o, const void *dO, const float *lse, const int32_t *block_idx,
                       void *dq, void *dk, void *dv, void *ws, size_t ws_bytes, void *stream);

/*
 * Dense causal attention (cuDNN-frontend page: the SDPA backward with
 * is_causal) as the special case where every row selects all of its blocks
 * 0..t/block_size.  Same arguments as the selection calls without an index;
 * p->S is ignored.
 */
nsa_status nsa_dense_causal_fwd(const nsa_problem *p, const void *q, const void *k,
                                const void *v, void *o, float *lse, void *ws, size_t ws_bytes,
                                void *stream);
nsa_status nsa_dense_causal_bwd(const nsa_problem *p, const void *q, const void *k,
                                const void *v, const void *o, const void *dO, const float *lse,
                                void *dq, void *dk, void *dv, void *ws, size_t ws_bytes,
                                void *stream);

/*
 * Packed variable-length selection attention (cuDNN-frontend page: the THD
 * path with cum_seqlen_q / cum_seqlen_k; here both are the same array).
 * p->layout must be NSA_LAYOUT_THD, p->B the number of sequences, p->T an
 * upper bound on every sequence length and p->total_tokens = cu_seqlens[B].
 */
nsa_status nsa_sel_varlen_fwd(const nsa_problem *p, const int32_t *cu_seqlens, const void *q,
                              const void *k, const void *v, const int32_t *block_idx, void *o,
                              float *lse, void *ws, size_t ws_bytes, void *stream);
nsa_status nsa_sel_varlen_bwd(const nsa_problem *p, const int32_t *cu_seqlens, const void *q,
                              const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, const int32_t *block_idx, void *dq, void *dk,
                              void *dv, void *ws, size_t ws_bytes, void *stream);

/*
 * Sliding-window causal attention (cuDNN-frontend page: the dense causal
 * SDPA backward's sliding-window option; NSA's sliding-window branch): the
 * dense causal case restricted to each row's `window` most recent keys,
 * k in (t - window, t].  window >= 1 (else NSA_ERR_INVALID_ARG); a window of
 * T or more is the dense causal case.  cu_seqlens is NULL for BHTD
 * (p->layout NSA_LAYOUT_BHTD) and the packed-row offsets for THD, where the
 * window applies within each sequence.  p->S is ignored; the workspaces are
 * the dense ones (nsa_fwd_workspace_size, nsa_bwd_workspace_size).
 */
nsa_status nsa_swa_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens,
                       const void *q, const void *k, const void *v, void *o, float *lse,
                       void *ws, size_t ws_bytes, void *stream);
nsa_status nsa_swa_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens,
                       const void *q, const void *k, const void *v, const void *o,
                       const void *dO, const float *lse, void *dq, void *dk, void *dv,
                       void *ws, size_t ws_bytes, void *stream);

/*
 * Dense causal attention with attention sinks (the cuDNN-frontend page's
 * backward chain ends in a dSink kernel; the page does not define the sink,
 * and the plainest reading is taken): one fp32 logit sinks[h] per query head
 * joins every row's softmax denominator and carries no value, so
 *   LSE_t = log( sum_k exp(s_tk) + exp(sinks[h]) ),  P_tk = exp(s_tk - LSE_t),
 *   O_t = sum_k P_tk v_k,  dsinks[h] = - sum_{b,t} exp(sinks[h] - LSE_t) D_t
 * with D_t = <dO_t, O_t>; dQ/dK/dV keep their form with this LSE.  window = 0
 * is plain causal, >= 1 the sliding window of nsa_swa_*.  cu_seqlens as for
 * nsa_swa_*.  sinks (device, Hq floats) is read, dsinks (device, Hq floats)
 * is written (overwritten, not accumulated).  The forward writes o and lse
 * with the sink included; the backward takes them as the forward wrote them.
 * Workspaces as for the dense entries.
 */
nsa_status nsa_sink_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const float *sinks,
                        const void *q, const void *k, const void *v, void *o, float *lse, void *ws,
                        size_t ws_bytes, void *stream);
nsa_status nsa_sink_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const float *sinks,
                        const void *q, const void *k, const void *v, const void *o, const void *dO,
                        const float *lse, void *dq, void *dk, void *dv, float *dsinks, void *ws,
                        size_t ws_bytes, void *stream);

/*
 * Dense causal attention whose keys have lengths of their own (cuDNN-frontend
 * page: the SDPA backward's THD path takes cum_seqlen_q and cum_seqlen_k,
 * and its causal mask comes aligned to the top-left corner or, with
 * causal_bottom_right, to the bottom-right one; both combine with the
 * sliding window).  For a sequence with Lq query rows and Lk keys, row t
 * sits at key position c_t = t (p->bottom_right = 0) or t + Lk - Lq
 * (p->bottom_right = 1) and attends key k iff k <= c_t, k < Lk and, with
 * window >= 1, c_t - k < window.  A row that attends nothing (bottom-right
 * with Lq > Lk: the first Lq - Lk rows) gets O = 0, LSE = -inf and no
 * gradient.
 * Layouts: BHTD q, o, dO, dq [B,Hq,T,D], k, v, dk, dv [B,Hkv,Tk,D] (Tk =
 * p->Tk, or T when 0), lse [B,Hq,T]; cu_seqlens_q and cu_seqlens_k NULL.
 * THD: q [total_tokens,Hq,D], k [total_keys,Hkv,D], lse [total_tokens,Hq];
 * cu_seqlens_q [B+1] (cu_seqlens_q[B] = p->total_tokens) and cu_seqlens_k
 * [B+1] (cu_seqlens_k[B] = p->total_keys), both device int32; p->T and
 * p->Tk bound every query and key length.  window = 0 is plain causal.
 * The workspaces come from nsa_causal_{fwd,bwd}_workspace_size; p->S is
 * ignored.  With Lq = Lk both alignments are the dense causal case.
 */
size_t nsa_causal_fwd_workspace_size(const nsa_problem *p);
size_t nsa_causal_bwd_workspace_size(const nsa_problem *p);
nsa_status nsa_causal_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, const void *q, const void *k, const void *v,
                          void *o, float *lse, void *ws, size_t ws_bytes, void *stream);
nsa_status nsa_causal_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, const void *q, const void *k, const void *v,
                          const void *o, const void *dO, const float *lse, void *dq, void *dk,
                          void *dv, void *ws, size_t ws_bytes, void *stream);

/*
 * Reusable backward plan.  The pages build nothing like it: it is the inverse
 * index of one block_idx tensor (block -> ascending list of the tokens that
 * selected it, see nsa_build_inverse_index) together with the dK/dV work
 * units cut from it, built once -- for example right after the selection is
 * made, next to the forward -- and read by any number of backward calls on
 * the same block_idx, which then skip the index build.
 *  - nsa_plan_size: bytes of device memory a plan of problem p needs
 *    (0 if p is not a valid selection problem).  The plan buffer is
 *    caller-owned, 256-byte aligned.
 *  - nsa_plan_build: checks the arguments, then on `stream` validates
 *    block_idx and writes the plan.  cu_seqlens is NULL for BHTD (p->layout
 *    NSA_LAYOUT_BHTD) and the packed-row offsets for THD.  Index errors are
 *    read with nsa_get_error(plan, ...); bad entries are left out.  Where
 *    the dQ tensor-core kernel runs (bf16, D = 128, 64-key blocks, G a
 *    multiple of 8, BHTD) the plan also holds its query tiles' block unions
 *    with the tiles' tokens grouped by shared blocks (a tile need not hold
 *    consecutive tokens: fewer blocks per tile), which the planned backward
 *    reads instead of building consecutive-token unions; the forward groups
 *    its tiles the same way on every call.
 *  - nsa_bwd_planned_workspace_size / nsa_sel_bwd_planned: the selection
 *    backward (nsa_sel_bwd, or nsa_sel_varlen_bwd when p->layout is THD and
 *    cu_seqlens is given) taking the index from `plan`, which must have been
 *    built from the same p, cu_seqlens and block_idx contents (not checked).
 *    The call only reads the plan, so calls sharing one plan may run at the
 *    same time (each with its own ws).  Returns NSA_ERR_INVALID_ARG for a
 *    NULL or misaligned plan.
 */
size_t nsa_plan_size(const nsa_problem *p);
nsa_status nsa_plan_build(const nsa_problem *p, const int32_t *cu_seqlens, const int32_t *block_idx,
                          void *plan, size_t plan_bytes, void *stream);
size_t nsa_bwd_planned_workspace_size(const nsa_problem *p);
nsa_status nsa_sel_bwd_planned(const nsa_problem *p, const int32_t *cu_seqlens, const void *q,
                               const void *k, const void *v, const void *o, const void *dO,
                               const float *lse, const int32_t *block_idx, const void *plan,
                               void *dq, void *dk, void *dv, void *ws, size_t ws_bytes,
                               void *stream);

/*
 * do_dot pre-pass (cuDNN-frontend page: the do_dot kernel of the backward
 * chain): delta_t = sum_d dO_td * O_td for every query row, in fp32, layout
 * of lse.  cu_seqlens is NULL for BHTD.
 */
nsa_status nsa_do_dot(const nsa_problem *p, const int32_t *cu_seqlens, const void *o,
                      const void *dO, float *delta, void *stream);

/*
 * Inverse index (block -> selecting tokens), the step the backward uses so
 * that dK/dV accumulate without atomics.  Canonical form: offsets has
 * nsa_inverse_index_offsets_len(p) entries, an exclusive scan over
 * (b, g, j) in lexicographic order with j < ceil(T / block_size); the list
 * of (b, g, j) holds every sequence-local token t whose row selects block j,
 * ascending.  rows must have room for (tokens * Hkv * S) entries, where
 * tokens is B*T (BHTD) or total_tokens (THD).  ws is a backward workspace.
 * Bad entries are skipped and reported through nsa_get_error.
 */
int64_t nsa_inverse_index_offsets_len(const nsa_problem *p);
nsa_status nsa_build_inverse_index(const nsa_problem *p, const int32_t *cu_seqlens,
                                   const int32_t *block_idx, int32_t *offsets, int32_t *rows,
                                   void *ws, size_t ws_bytes, void *stream);

/*
 * nsa_build_inverse_index without a caller workspace.  The pages describe
 * nothing like it; it exists for callers that cannot allocate device memory
 * when they call in -- for example a runtime whose memory is carved up once
 * at start-up and may not grow afterwards, or code running where a
 * cudaMalloc would stall or break the surrounding stream schedule.  Same
 * arguments and results as nsa_build_inverse_index, except:
 *  - the scratch is a 2 MiB array inside the library (every GPU that loads
 *    the library holds it until the process exits).  A problem whose
 *    scratch would not fit -- 256 + 12 * B*Hkv*ceil(T/block_size) bytes plus
 *    32 bytes per dK/dV work unit, each part rounded up to 256 bytes --
 *    returns NSA_ERR_UNSUPPORTED before any launch;
 *  - the first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before
 *    any stream capture;
 *  - every call uses the same array and the call clears what must start at
 *    zero, so calls that can overlap on the GPU (other streams, other host
 *    threads) race and must not be issued;
 *  - device-side index errors are copied into *status_out (device int32,
 *    4-byte aligned, may be NULL) on `stream` instead of a workspace error
 *    word;
 *  - the array's device address is looked up once per device and kept for
 *    the life of the process: after cudaDeviceReset (or anything else that
 *    destroys the device's primary context) this entry point must not be
 *    called again in that process.
 * Nothing is allocated or freed.
 */
nsa_status nsa_build_inverse_index_noalloc(const nsa_problem *p, const int32_t *cu_seqlens,
                                           const int32_t *block_idx, int32_t *offsets,
                                           int32_t *rows, int32_t *status_out, void *stream);

/*
 * Self-test of the device-side timeout path (instrumentation, off by
 * default; not thread-safe).  Every wait inside the tensor-core kernels is
 * bounded: a wait that runs out makes the kernel stop its work, wait (again
 * bounded) for its own copies and products in flight, free its tensor
 * memory, and report NSA_ERR_DEVICE_TIMEOUT through the workspace error word,
 * leaving the CUDA context usable.  nsa_debug_stall(kernel, wait_limit_us)
 * lets a test run that path without any fault: while `kernel` is 1 (the
 * forward), 2 (the dK/dV kernel) or 3 (the dQ kernel), that kernel is
 * launched with the thread that issues its S = Q K^T products idle, so the
 * first wait on S runs out; `wait_limit_us` (1 .. 2000000; 0 = the default
 * of 2 s) replaces the limit of every tensor-core kernel's waits.
 * nsa_debug_stall(0, 0) restores normal operation.  Returns
 * NSA_ERR_INVALID_ARG for values out of range.  The CUDA-core kernels (fp32,
 * other head dims and block sizes) have no waits and ignore it.
 */
nsa_status nsa_debug_stall(int32_t kernel, int32_t wait_limit_us);

/*
 * The step that PRODUCES the index: NSA's block selection.  The pages take
 * idx as given (the gradcheck-gate page names "NSA selection" and builds
 * idx with a helper it does not print), so this is the plainest reading of
 * the selection step, consistent with the pages' tests (slot 0 = the row's
 * own block):
 *   block j of a sequence is complete at row t  iff  (j+1)*block_size - 1 <= t
 *   p[h,t,j]    = softmax over the blocks j complete at t of scale*<q[h,t], kc[g,j]>
 *   score[g,t,j] = sum over the G query heads h of kv head g of p[h,t,j]
 *                  (0 for blocks not complete at t)
 *   idx[g,t]    = [ t / block_size, then the S - 1 blocks other than it that
 *                   are complete at t with the largest scores, in decreasing
 *                   order (equal scores: smaller j first; NaN ranks as
 *                   -infinity), then -1 for the slots left ]
 * kc is one compressed key per block and kv head; NSA learns that
 * compression, so kc is an input.  nsa_compress_keys_mean writes the
 * weight-free stand-in (the mean of the block's keys).
 *
 * These entries take either layout: p->layout THD with cu_seqlens (block ids
 * and causality local to each sequence), else BHTD with cu_seqlens NULL.
 *   kc      [B, Hkv, nb, D] dense, the problem's dtype, nb = ceil(T /
 *           block_size) (THD: T bounds every sequence length); rows of blocks
 *           not complete in their sequence are zero (compress) or unused
 *   scores  float, [B, Hkv, T, nb] (BHTD) or [total, Hkv, nb] (THD): the
 *           index's rows, nb scores each
 *   idx     int32, the index layout ([B, Hkv, T, S] / [total, Hkv, S])
 * k honours p->kv_stride and q p->q_stride; kc, scores and idx are dense.
 * Pointers are device pointers owned by the caller: q, k and kc 16-byte
 * aligned, scores and idx 4-byte aligned.  Shape errors are returned before
 * any launch.  nsa_block_scores runs on the tensor cores (bf16; fp32 by
 * split precision; D in {32, 64, 128}) with bounded waits: its workspace
 * (nsa_select_workspace_size bytes, 256-byte aligned) carries the device
 * error word read by nsa_get_error.  nsa_compress_keys_mean and
 * nsa_select_topk report no device errors and take no workspace.
 */
size_t nsa_select_workspace_size(const nsa_problem *p);
nsa_status nsa_compress_keys_mean(const nsa_problem *p, const int32_t *cu_seqlens, const void *k, void *kc,
                                  void *stream);
nsa_status nsa_block_scores(const nsa_problem *p, const int32_t *cu_seqlens, const void *q, const void *kc,
                            float *scores, void *ws, size_t ws_bytes, void *stream);
nsa_status nsa_select_topk(const nsa_problem *p, const int32_t *cu_seqlens, const float *scores, int32_t *idx,
                           void *stream);

/*
 * Reads the device error word of a workspace used by the calls above,
 * after synchronising `stream`, into *out (an nsa_status value), and clears
 * it.  Returns NSA_ERR_CUDA if the read itself fails.
 */
nsa_status nsa_get_error(void *ws, void *stream, int32_t *out);

/* Static string naming a status. */
const char *nsa_status_string(int32_t status);

/* Number of (query row, attended key) pairs summed over query heads; the
 * unit of the effective-FLOP count (10*D per pair for the backward).
 * Computed on the device into *out_pairs (device int64), on `stream`. */
nsa_status nsa_count_pairs(const nsa_problem *p, const int32_t *cu_seqlens,
                           const int32_t *block_idx, int64_t *out_pairs, void *stream);

/*
 * Per-kernel timing (instrumentation, off by default).  nsa_trace_enable(n)
 * creates n pairs of CUDA events (n <= 0 destroys them and turns timing
 * off); while on, every kernel an entry point launches is bracketed by an
 * event pair on the call's stream, until n launches have been recorded.
 * nsa_trace_get(i, ...) waits for launch i to finish and returns the kernel
 * name (static string) and its duration in milliseconds.  Not thread-safe:
 * use from one host thread.
 */
nsa_status nsa_trace_enable(int32_t max_records);
void nsa_trace_reset(void);
int32_t nsa_trace_count(void);
nsa_status nsa_trace_get(int32_t i, const char **name, float *ms);

#ifdef __cplusplus
}
#endif

#endif /* NSA_H */
