// nsa_api.cu -- the C ABI of libnsa.so (include/nsa.h): argument checks,
// workspace carving and the launch sequence of each entry point.  No entry
// point allocates memory or synchronises; all work is ordered on the
// caller's stream (a launch that may run beside it goes on a helper stream
// forked from and joined back to it by events).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "launch.h"

using namespace nsa;

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// SPARSE: selection; DENSE: every block up to the diagonal (queries and keys
// of equal length); CAUSAL: dense with the keys' own lengths and the diagonal
// aligned top-left or bottom-right (nsa_causal_*)
enum Mode { SPARSE = 0, DENSE = 1, CAUSAL = 2 };

// One tensor's declared (batch, head, token) strides into `out`: all zero
// selects the dense layout with H heads; otherwise every stride in use must
// be positive, a multiple of 16 bytes and below 2^40 bytes (the tensor-map
// limits).  THD ignores the batch entry.
bool take_strides(const int64_t in[3], const nsa_problem *p, bool thd, int H, int T, Strides &out)
{
    const int64_t D = p->D, es = p->dtype == NSA_DTYPE_BF16 ? 2 : 4;
    if (in[0] == 0 && in[1] == 0 && in[2] == 0) {
        out = thd ? Strides{0, D, (int64_t)H * D} : Strides{(int64_t)H * T * D, (int64_t)T * D, D};
        return true;
    }
    for (int i = thd ? 1 : 0; i < 3; ++i)
        if (in[i] <= 0 || (in[i] * es) % 16 != 0 || in[i] * es >= ((int64_t)1 << 40))
            return false;
    out = Strides{thd ? 0 : in[0], in[1], in[2]};
    return true;
}

// Checks the problem and fills the device geometry.  `want_thd` is the
// layout the entry point requires.
nsa_status make_geo(const nsa_problem *p, bool want_thd, Mode mode, const int32_t *cu, Geo &g, int window = 0,
                    const int32_t *cuk = nullptr)
{
    if (window < 0 || (window > 0 && mode == SPARSE))
        return NSA_ERR_INVALID_ARG;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    // the keys' geometry: their own for the causal entries, else the queries'
    const bool own_keys = mode == CAUSAL;
    if (own_keys && (p->Tk < 0 || p->total_keys < 0 || (p->bottom_right != 0 && p->bottom_right != 1) ||
                     (want_thd && (!cuk || p->total_keys < 1))))
        return NSA_ERR_INVALID_ARG;
    const int Tk = own_keys && p->Tk > 0 ? p->Tk : p->T;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->T < 1)
        return NSA_ERR_INVALID_ARG;
    if (p->Hq % p->Hkv != 0)
        return NSA_ERR_INVALID_ARG;
    if (p->dtype != NSA_DTYPE_F32 && p->dtype != NSA_DTYPE_BF16)
        return NSA_ERR_INVALID_ARG;
    if (p->layout != (want_thd ? NSA_LAYOUT_THD : NSA_LAYOUT_BHTD))
        return NSA_ERR_INVALID_ARG;
    if (mode == SPARSE && p->S < 1)
        return NSA_ERR_INVALID_ARG;
    if (p->D != 32 && p->D != 64 && p->D != 128)
        return NSA_ERR_UNSUPPORTED;
    if (p->block_size != 16 && p->block_size != 32 && p->block_size != 64)
        return NSA_ERR_UNSUPPORTED;
    if (mode == SPARSE && p->S > 256)
        return NSA_ERR_UNSUPPORTED;
    if (want_thd) {
        if (!cu || p->total_tokens < 0)
            return NSA_ERR_INVALID_ARG;
    }
    const int64_t ntok = want_thd ? (int64_t)p->total_tokens : (int64_t)p->B * p->T;
    if (ntok * p->Hq * (int64_t)p->D >= ((int64_t)1 << 40))
        return NSA_ERR_UNSUPPORTED;
    // the index-side sizes (list entries, per-block counters, work units) are
    // held in int: refuse problems whose counts would not fit
    const int64_t ntok_k = !own_keys ? ntok : want_thd ? (int64_t)p->total_keys : (int64_t)p->B * Tk;
    if (ntok_k * p->Hkv * (int64_t)p->D >= ((int64_t)1 << 40))
        return NSA_ERR_UNSUPPORTED;
    const int64_t nb = (Tk + p->block_size - 1) / p->block_size;
    if (ntok >= INT32_MAX || ntok_k >= INT32_MAX || ntok * p->Hq >= INT32_MAX ||
        (int64_t)p->B * p->Hkv * nb >= INT32_MAX)
        return NSA_ERR_UNSUPPORTED;
    if (mode == SPARSE && ntok * p->Hkv * p->S >= INT32_MAX)  // inverse-index entries
        return NSA_ERR_UNSUPPORTED;
    memset(&g, 0, sizeof(g));
    g.B = p->B;
    g.Hq = p->Hq;
    g.Hkv = p->Hkv;
    g.G = p->Hq / p->Hkv;
    g.T = p->T;
    g.D = p->D;
    g.bs = p->block_size;
    g.nbmax = (int)nb;  // key blocks of the longest key sequence
    g.S = mode != SPARSE ? g.nbmax : p->S;
    g.ntok = (int)ntok;
    g.thd = want_thd ? 1 : 0;
    g.dense = mode != SPARSE ? 1 : 0;
    g.Tk = Tk;
    g.ntok_k = (int)ntok_k;
    g.cuk = own_keys && want_thd ? cuk : cu;
    g.br = own_keys ? p->bottom_right : 0;
    g.window = window;
    g.scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->D);
    g.scale_l2 = g.scale * 1.4426950408889634f;
    g.cu = cu;
    if (!take_strides(p->q_stride, p, want_thd, p->Hq, p->T, g.sq) ||
        !take_strides(p->kv_stride, p, want_thd, p->Hkv, Tk, g.skv) ||
        !take_strides(p->o_stride, p, want_thd, p->Hq, p->T, g.so) ||
        !take_strides(p->dq_stride, p, want_thd, p->Hq, p->T, g.sdq) ||
        !take_strides(p->dkv_stride, p, want_thd, p->Hkv, Tk, g.sdkv))
        return NSA_ERR_INVALID_ARG;
    // the row-gather maps of q and o fold the batch into the token index when
    // it does not fold into the head index (a packed [B, T, H, D] tensor)
    auto bt = [&](const Strides &st, int H) {
        return !want_thd && p->B > 1 && st.b != (int64_t)H * st.h && st.b == (int64_t)p->T * st.t;
    };
    g.q_bt = bt(g.sq, p->Hq);
    g.o_bt = bt(g.so, p->Hq);
    Strides dense_o;
    const int64_t zero[3] = {0, 0, 0};
    take_strides(zero, p, want_thd, p->Hq, p->T, dense_o);
    g.o_lin = (want_thd || g.so.b == dense_o.b) && g.so.h == dense_o.h && g.so.t == dense_o.t;
    return NSA_OK;
}

// Backward plan: the inverse index of one block_idx and its dK/dV work
// units, in one region that starts with a header (n_units, index errors):
// header | counts | offsets | unit list | per-block chunk count and partial
// slot | per-chunk histograms (chunked build) | token lists (sparse only).
struct PlanLayout {
    size_t counts, offsets, units, nchunk, slot, chunkc, rows, utable, total;
    int chunk, max_units;
    bool has_utable;  // the plan also holds the query-tile unions, tiles grouped by shared blocks
};

int tiles_tokens(const Geo &g) { return g.G >= 128 ? 1 : 128 / g.G; }

// dtype >= 0 (a plan built by nsa_plan_build): where the tensor-core kernels
// take a grouped union table, the plan ends with one
PlanLayout plan_layout(const Geo &g, int dtype = -1)
{
    PlanLayout w;
    const int64_t nbgj = (int64_t)g.B * g.Hkv * g.nbmax;
    // tokens per dK/dV unit: 128 row tiles of the tensor-core kernel (longer
    // units mean fewer accumulator drains and split-block partials; the dQ
    // kernel launched behind dK/dV takes the SMs its uneven end leaves); 4 row
    // tiles for the other shapes' kernel, whose CTA walks its unit's tiles one
    // after another (the longest unit sets its time)
    w.chunk = tiles_tokens(g) * (g.D == 128 && g.bs == 64 ? 128 : 4);
    // upper bound on list entries; dense: a row of sequence-local token t
    // attends t/bs + 1 <= nbmax/2 + 1 blocks on average over a sequence, or
    // with keys of their own lengths (a short query run at the end of long
    // keys) up to every block
    const bool own_keys = g.br || g.Tk != g.T || g.cuk != g.cu;
    const int64_t sel_total = !g.dense ? (int64_t)g.ntok * g.Hkv * g.S
                              : own_keys ? (int64_t)g.ntok * g.Hkv * g.nbmax
                                         : (int64_t)g.ntok * g.Hkv * (g.nbmax / 2 + 1);
    w.max_units = (int)(nbgj + (sel_total + w.chunk - 1) / w.chunk);
    size_t off = kAlign;  // header
    w.counts = off;
    off = align_up(off + sizeof(int) * (size_t)nbgj);
    w.offsets = off;
    off = align_up(off + sizeof(int) * (size_t)(nbgj + 1));
    w.units = off;
    off = align_up(off + sizeof(Unit) * (size_t)w.max_units);
    w.nchunk = off;
    off = align_up(off + sizeof(int) * (size_t)nbgj);
    w.slot = off;
    off = align_up(off + sizeof(int) * (size_t)nbgj);
    w.chunkc = off;
    if (!g.dense && csr_chunked_ok(g))
        off = align_up(off + sizeof(int) * (size_t)nbgj * csr_nchunks(g));
    w.rows = off;
    if (!g.dense)
        off = align_up(off + sizeof(int) * (size_t)g.ntok * g.Hkv * g.S);
    w.utable = off;
    w.has_utable = dtype >= 0 && !g.dense && tc_supported(g, dtype) && qtile_groupable(g) &&
                   qtile_union_table_bytes(g) > 0;
    if (w.has_utable)
        off = align_up(off + qtile_union_table_bytes(g));
    w.total = off;
    return w;
}

// Backward workspace: header (error word) | delta fp32 [rows] | fp32 dK/dV
// partials (tensor-core path) | the plan, unless the call is given one.
struct BwdWs {
    size_t delta, partials, utable, plan, total;
    PlanLayout pl;
};

BwdWs bwd_layout(const Geo &g, int dtype)
{
    BwdWs w;
    w.pl = plan_layout(g);
    size_t off = kAlign;
    w.delta = off;
    off = align_up(off + sizeof(float) * (size_t)g.ntok * g.Hq);
    w.partials = off;
    if (tc_supported(g, dtype) || gtc_supported(g, dtype))
        off = align_up(off + sizeof(float) * 2 * (size_t)g.bs * g.D * (size_t)w.pl.max_units);
    w.utable = off;  // the dQ kernel's query-tile unions
    if (tc_supported(g, dtype))
        off = align_up(off + qtile_union_table_bytes(g));
    w.plan = off;
    w.total = off + w.pl.total;
    return w;
}

inline nsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NSA_OK : NSA_ERR_CUDA; }

#define NSA_TRY(expr)                                  \
    do {                                               \
        cudaError_t _e = (expr);                       \
        if (_e != cudaSuccess)                         \
            return NSA_ERR_CUDA;                       \
    } while (0)

// ---- opt-in per-kernel timing (nsa_trace_*): an event pair around every
// kernel launch, recorded on the launch stream.  Off unless enabled.
struct TraceRec {
    const char *name;
    cudaEvent_t start, stop;
};
TraceRec *g_trace = nullptr;
int g_trace_cap = 0, g_trace_n = 0;

struct TraceScope {
    TraceRec *rec = nullptr;
    cudaStream_t st;
    TraceScope(const char *name, cudaStream_t s) : st(s)
    {
        if (g_trace && g_trace_n < g_trace_cap) {
            rec = &g_trace[g_trace_n++];
            rec->name = name;
            cudaEventRecord(rec->start, st);
        }
    }
    ~TraceScope()
    {
        if (rec)
            cudaEventRecord(rec->stop, st);
    }
};

#define NSA_LAUNCH(name, expr)                         \
    do {                                               \
        TraceScope _ts(name, st);                      \
        NSA_TRY(expr);                                 \
    } while (0)

// ---- a helper stream per device, for a launch that can run beside the
// ones that follow it on the caller's stream (the other-shapes dQ needs
// only delta, so it runs beside the index build and dK/dV).  Created on
// first use; kept for the process.
struct Helper {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;  // held from a fork to its join: the two events are shared
};
constexpr int kMaxDevices = 64;
Helper g_helpers[kMaxDevices];
std::mutex g_helpers_mu;

Helper *helper_of_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_helpers_mu);
    Helper &h = g_helpers[dev];
    if (!h.s) {
        cudaStream_t s = nullptr;
        cudaEvent_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
            if (s)
                cudaStreamDestroy(s);
            if (a)
                cudaEventDestroy(a);
            (void)cudaGetLastError();
            return nullptr;
        }
        h.fork = a;
        h.join = b;
        h.s = s;
    }
    return &h;
}

// begin(): work launched on side() from here on starts after everything
// enqueued on st so far; join() (or scope exit) makes what st enqueues next
// wait for it.  Without a helper (or before begin) side() is st itself: the
// launches stay in order.
struct Fork {
    cudaStream_t st;
    Helper *h = nullptr;
    bool forked = false, joined = false;
    std::unique_lock<std::mutex> lk;
    explicit Fork(cudaStream_t s) : st(s) {}
    void begin()
    {
        if (forked || !(h = helper_of_current_device()))
            return;
        lk = std::unique_lock<std::mutex>(h->mu);
        forked = cudaEventRecord(h->fork, st) == cudaSuccess && cudaStreamWaitEvent(h->s, h->fork, 0) == cudaSuccess;
        if (!forked) {
            (void)cudaGetLastError();
            lk.unlock();
        }
    }
    cudaStream_t side() const { return forked && !joined ? h->s : st; }
    void join()
    {
        if (!forked || joined)
            return;
        if (cudaEventRecord(h->join, h->s) != cudaSuccess || cudaStreamWaitEvent(st, h->join, 0) != cudaSuccess)
            cudaStreamSynchronize(h->s);  // the join failed: order by waiting instead
        joined = true;
        lk.unlock();
    }
    ~Fork() { join(); }
};

nsa_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws || ((uintptr_t)ws & (kAlign - 1)) || ws_bytes < need)
        return NSA_ERR_WORKSPACE;
    return NSA_OK;
}

// workspace bytes of a forward / backward of this mode (0: invalid problem)
size_t fwd_ws_need(const nsa_problem *p, Mode mode);
size_t bwd_ws_need(const nsa_problem *p, Mode mode);

nsa_status run_fwd(const nsa_problem *p, bool thd, Mode mode, const int32_t *cu, const void *q,
                   const void *k, const void *v, const int32_t *idx, void *o, float *lse,
                   void *ws, size_t ws_bytes, void *stream, int window = 0, const float *sinks = nullptr,
                   const int32_t *cuk = nullptr)
{
    Geo g;
    nsa_status s = make_geo(p, thd, mode, cu, g, window, cuk);
    if (s != NSA_OK)
        return s;
    if (!q || !k || !v || !o || !lse || (mode == SPARSE && !idx))
        return NSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return NSA_ERR_INVALID_ARG;
    if ((s = check_ws(ws, ws_bytes, fwd_ws_need(p, mode))) != NSA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    WsHeader *hdr = (WsHeader *)ws;
    NSA_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
    if (g.ntok == 0)
        return NSA_OK;
    if (mode == SPARSE)
        NSA_LAUNCH("validate_index", launch_validate_index(g, idx, &hdr->err, st));
    if (tc_supported(g, p->dtype)) {
        // the query-tile unions (sparse only), alongside the validation
        int *utable = mode == SPARSE && qtile_union_table_bytes(g) ? (int *)((char *)ws + kAlign) : nullptr;
        if (utable)
            NSA_LAUNCH("qtile_unions", launch_qtile_unions(g, idx, utable, st, true));
        NSA_LAUNCH("fwd_tc",
                   launch_fwd_tc(g, q, k, v, idx, utable, utable && qtile_groupable(g), o, lse, &hdr->err,
                                 &hdr->tile_next, mode == SPARSE, st));
    }
    else if (gtc_supported(g, p->dtype))
        NSA_LAUNCH("fwd_gtc", launch_fwd_gtc(g, q, k, v, idx, o, lse, p->dtype, &hdr->err, st));
    else
        NSA_LAUNCH("fwd_simt", launch_fwd_simt(g, q, k, v, idx, o, lse, p->dtype, st));
    if (sinks)
        NSA_LAUNCH("sink_fwd", launch_sink_fwd(g, sinks, o, lse, p->dtype, st));
    return NSA_OK;
}

// the inverse index into (offsets, rows); counts is scratch of nbgj ints
// chunk_counts (nullable) selects the chunked build: per-chunk histograms
// and an ordered per-chunk fill; otherwise one atomic count pass and one
// ordered walk per block list.  Both give the same canonical lists.
// dot (nullable, chunked build only): delta computed in the count's launch
// fork (nullable, with dot): begun once the count's launch (and so delta)
// is enqueued; join (nullable): joined before the fill
nsa_status build_csr(const Geo &g, const int32_t *idx, int *counts, int *offsets, int *rows,
                     Unit *units, int *nchunk, int *slot, WsHeader *hdr, int *err, int chunk, cudaStream_t st,
                     int *chunk_counts = nullptr, const DotArgs *dot = nullptr, Fork *fork = nullptr,
                     Fork *join = nullptr)
{
    const size_t nbgj = (size_t)g.B * g.Hkv * g.nbmax;
    if (!g.dense && chunk_counts && csr_chunked_ok(g)) {
        NSA_LAUNCH(dot ? "do_dot+csr_count" : "csr_count",
                   launch_csr_chunk_count(g, idx, chunk_counts, counts, err, st, dot));
        if (dot && fork)
            fork->begin();
        NSA_LAUNCH("csr_scan", launch_csr_scan(g, counts, offsets, units, nchunk, slot, hdr, chunk, st));
        if (join)
            join->join();
        NSA_LAUNCH("csr_fill", launch_csr_chunk_fill(g, idx, chunk_counts, offsets, rows, st));
        return NSA_OK;
    }
    if (!g.dense) {
        NSA_TRY(cudaMemsetAsync(counts, 0, sizeof(int) * nbgj, st));
        NSA_LAUNCH("csr_count", launch_csr_count(g, idx, counts, err, st));
    }
    NSA_LAUNCH("csr_scan", launch_csr_scan(g, counts, offsets, units, nchunk, slot, hdr, chunk, st));
    if (join)
        join->join();
    if (!g.dense)
        NSA_LAUNCH("csr_fill", launch_csr_fill(g, idx, offsets, rows, st));
    return NSA_OK;
}

// Builds the plan of `idx` at `plan8` (layout L); index errors go to *err.
// With dot, delta is computed in the same pass (see build_csr).
nsa_status build_plan(const Geo &g, const int32_t *idx, char *plan8, const PlanLayout &L, int *err, cudaStream_t st,
                      const DotArgs *dot = nullptr, Fork *fork = nullptr, Fork *join = nullptr)
{
    WsHeader *phdr = (WsHeader *)plan8;
    NSA_TRY(cudaMemsetAsync(phdr, 0, sizeof(WsHeader), st));
    return build_csr(g, idx, (int *)(plan8 + L.counts), (int *)(plan8 + L.offsets), (int *)(plan8 + L.rows),
                     (Unit *)(plan8 + L.units), (int *)(plan8 + L.nchunk), (int *)(plan8 + L.slot), phdr, err,
                     L.chunk, st, (int *)(plan8 + L.chunkc), dot, fork, join);
}

// whether build_plan takes the chunked path (which can carry the dot)
bool plan_is_chunked(const Geo &g) { return !g.dense && csr_chunked_ok(g); }

nsa_status run_bwd(const nsa_problem *p, bool thd, Mode mode, const int32_t *cu, const void *q,
                   const void *k, const void *v, const void *o, const void *dO, const float *lse,
                   const int32_t *idx, const void *plan, void *dq, void *dk, void *dv, void *ws,
                   size_t ws_bytes, void *stream, int window = 0, const float *sinks = nullptr,
                   float *dsinks = nullptr, const int32_t *cuk = nullptr)
{
    Geo g;
    nsa_status s = make_geo(p, thd, mode, cu, g, window, cuk);
    if (s != NSA_OK)
        return s;
    if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || (mode == SPARSE && !idx))
        return NSA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void *x : ptrs)
        if (!aligned16(x))
            return NSA_ERR_INVALID_ARG;
    if (plan && ((uintptr_t)plan & (kAlign - 1)))
        return NSA_ERR_INVALID_ARG;
    const BwdWs L = bwd_layout(g, p->dtype);
    if ((s = check_ws(ws, ws_bytes, plan ? L.plan : bwd_ws_need(p, mode))) != NSA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    char *w8 = (char *)ws;
    WsHeader *hdr = (WsHeader *)ws;
    char *pl8 = plan ? (char *)plan : w8 + L.plan;
    const PlanLayout &P = L.pl;
    // a plan built by nsa_plan_build may end with the grouped union table
    const PlanLayout PP = plan ? plan_layout(g, p->dtype) : L.pl;
    float *delta = (float *)(w8 + L.delta);
    float *partials = (float *)(w8 + L.partials);
    const int *offsets = (const int *)(pl8 + P.offsets);
    const int *rows = (const int *)(pl8 + P.rows);
    const Unit *units = (const Unit *)(pl8 + P.units);
    const int *nchunk = (const int *)(pl8 + P.nchunk);
    const int *slot = (const int *)(pl8 + P.slot);
    const WsHeader *phdr = (const WsHeader *)pl8;
    NSA_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
    if (g.ntok == 0) {
        if (sinks)
            NSA_TRY(cudaMemsetAsync(dsinks, 0, sizeof(float) * g.Hq, st));
        return NSA_OK;
    }
    // delta = rowsum(dO * O): in the index count's launch when the index is
    // built here by chunks, else on its own
    const DotArgs dot{o, dO, delta, p->dtype};
    const bool fused = !plan && plan_is_chunked(g);
    // the other-shapes dQ reads only delta (not the inverse index): it runs
    // on a helper stream beside the index build and dK/dV, which leave SMs
    // free (one CTA of ~170 registers a thread per query tile)
    const bool gtc = !tc_supported(g, p->dtype) && gtc_supported(g, p->dtype);
    Fork fork(st);
    // The dQ tensor-core kernel's union table with tiles grouped by shared
    // blocks: built on the helper stream beside delta and the index build
    // (it reads only the index), joined before the fill; its table is read
    // only by dQ, after dK/dV.
    Fork gfork(st);
    bool grouped = false;
    if (tc_supported(g, p->dtype) && !plan && mode == SPARSE && qtile_groupable(g) && qtile_union_table_bytes(g)) {
        gfork.begin();
        if (gfork.forked) {
            const cudaStream_t st = gfork.side();
            // (64-token windows: grouping over 96 or 128 outlasts the work it runs
            // beside and delays the fill)
            NSA_LAUNCH("qtile_unions", launch_qtile_unions(g, idx, (int *)(w8 + L.utable), st, true, 2));
            grouped = true;
        }
    }
    if (!fused)
        NSA_LAUNCH("do_dot", launch_do_dot(g, o, dO, delta, p->dtype, st));
    if (gtc && !fused)
        fork.begin();
    if (!plan && (s = build_plan(g, idx, pl8, P, &hdr->err, st, fused ? &dot : nullptr, gtc ? &fork : nullptr,
                                 grouped ? &gfork : nullptr)) != NSA_OK)
        return s;
    gfork.join();
    if (tc_supported(g, p->dtype)) {
        // the query-tile unions (sparse only): grouped and built beside the
        // index build above, or a plan's (built once), or else of consecutive
        // tokens, built here alongside the kernel before (they read only the
        // index)
        int *utable = qtile_union_table_bytes(g) ? (int *)(w8 + L.utable) : nullptr;
        if (PP.has_utable)
            utable = (int *)(pl8 + PP.utable);
        else if (utable && !grouped)
            NSA_LAUNCH("qtile_unions", launch_qtile_unions(g, idx, utable, st, false));
        NSA_LAUNCH("dkdv_tc", launch_dkdv_tc(g, q, k, v, dO, lse, delta, offsets, rows, units, phdr, P.max_units,
                               partials, dk, dv, &hdr->err, st));
        // dQ right after dK/dV: it is that kernel's programmatic dependent
        NSA_LAUNCH("dq_tc",
                   launch_dq_tc(g, q, k, v, dO, lse, delta, idx, utable, PP.has_utable || grouped, dq, &hdr->err,
                                &hdr->tile_next, st));
        NSA_LAUNCH("dkdv_reduce", launch_dkdv_reduce(g, nchunk, slot, partials, dk, dv, p->dtype, st));
    } else if (gtc) {
        {
            const cudaStream_t st = fork.side();
            NSA_LAUNCH("dq_gtc", launch_dq_gtc(g, q, k, v, dO, lse, delta, idx, dq, p->dtype, &hdr->err, st));
        }
        NSA_LAUNCH("dkdv_gtc", launch_dkdv_gtc(g, q, k, v, dO, lse, delta, offsets, rows, units, phdr, P.max_units,
                                               partials, dk, dv, p->dtype, &hdr->err, st));
        // a programmatic dependent of dK/dV (it waits for it before reading)
        NSA_LAUNCH("dkdv_reduce", launch_dkdv_reduce(g, nchunk, slot, partials, dk, dv, p->dtype, st, true));
    } else {
        NSA_LAUNCH("dkdv_simt", launch_dkdv_simt(g, q, k, v, dO, lse, delta, offsets, rows, dk, dv, p->dtype, st));
        NSA_LAUNCH("dq_simt", launch_dq_simt(g, q, k, v, dO, lse, delta, idx, dq, p->dtype, st));
    }
    if (sinks)
        NSA_LAUNCH("sink_bwd", launch_sink_bwd(g, sinks, lse, delta, dsinks, st));
    return NSA_OK;
}

WaitTest g_wait_test = {WAIT_TEST_NONE, 0};

// stand-ins for device pointers in the size queries (never dereferenced):
// distinct, so that a packed causal problem's keys count as their own
const int32_t *const kFakeCuQ = (const int32_t *)16, *const kFakeCuK = (const int32_t *)32;

// The selection-step entries take either layout (THD when p->layout says so,
// with cu_seqlens); index rows and block scores follow the index's layout.
nsa_status select_geo(const nsa_problem *p, const int32_t *cu_seqlens, Geo &g, Mode mode)
{
    if (!p)
        return NSA_ERR_INVALID_ARG;
    return make_geo(p, p->layout == NSA_LAYOUT_THD, mode, cu_seqlens, g);
}

size_t fwd_ws_need(const nsa_problem *p, Mode mode)
{
    if (mode != CAUSAL)
        return nsa_fwd_workspace_size(p);
    Geo g;
    const bool thd = p && p->layout == NSA_LAYOUT_THD;
    return make_geo(p, thd, CAUSAL, thd ? kFakeCuQ : nullptr, g, 0, thd ? kFakeCuK : nullptr) == NSA_OK ? kAlign : 0;
}

size_t bwd_ws_need(const nsa_problem *p, Mode mode)
{
    if (mode != CAUSAL)
        return nsa_bwd_workspace_size(p);
    Geo g;
    const bool thd = p && p->layout == NSA_LAYOUT_THD;
    if (make_geo(p, thd, CAUSAL, thd ? kFakeCuQ : nullptr, g, 0, thd ? kFakeCuK : nullptr) != NSA_OK)
        return 0;
    return bwd_layout(g, p->dtype).total;
}

}  // namespace

WaitTest nsa::wait_test() { return g_wait_test; }

// ---- scratch for nsa_build_inverse_index_noalloc --------------------------
// Some callers cannot allocate device memory at call time (see include/nsa.h),
// so this one entry point keeps its scratch in a fixed array that every GPU
// loading the library holds until the process exits.
constexpr size_t kNoallocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char nsa_noalloc_scratch[kNoallocScratchBytes];

namespace {

// Device address of nsa_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name only stands in for the symbol;
// handing it to a kernel directly would use the wrong memory.
nsa_status noalloc_scratch_address(void **out)
{
    static void *addr[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NSA_ERR_CUDA;
    if (dev < 0 || dev >= 128)
        return NSA_ERR_UNSUPPORTED;
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, nsa_noalloc_scratch) != cudaSuccess || !p)
            return NSA_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return NSA_OK;
}

}  // namespace

extern "C" {

size_t nsa_fwd_workspace_size(const nsa_problem *p)
{
    Geo g;
    if (!p)
        return 0;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    // dense and sparse forwards share the layout: the header, then (sparse,
    // tensor-core path) the query-tile union table
    if (make_geo(p, thd, SPARSE, thd ? (const int32_t *)16 : nullptr, g) == NSA_OK)
        return kAlign + (tc_supported(g, p->dtype) ? align_up(qtile_union_table_bytes(g)) : 0);
    if (make_geo(p, thd, DENSE, thd ? (const int32_t *)16 : nullptr, g) != NSA_OK)
        return 0;
    return kAlign;
}

size_t nsa_bwd_workspace_size(const nsa_problem *p)
{
    Geo g;
    if (!p)
        return 0;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    const int32_t *fake_cu = thd ? (const int32_t *)16 : nullptr;
    if (make_geo(p, thd, SPARSE, fake_cu, g) == NSA_OK) {
        // the dense entry uses S = nbmax; size for the larger of the two
        Geo gd;
        make_geo(p, thd, DENSE, fake_cu, gd);
        const size_t sa = bwd_layout(g, p->dtype).total, sb = bwd_layout(gd, p->dtype).total;
        return sa > sb ? sa : sb;
    }
    if (make_geo(p, thd, DENSE, fake_cu, g) == NSA_OK)
        return bwd_layout(g, p->dtype).total;
    return 0;
}

size_t nsa_sel_fwd_workspace_size(const nsa_problem *p) { return nsa_fwd_workspace_size(p); }
size_t nsa_sel_bwd_workspace_size(const nsa_problem *p) { return nsa_bwd_workspace_size(p); }

nsa_status nsa_sel_fwd(const nsa_problem *p, const void *q, const void *k, const void *v,
                       const int32_t *block_idx, void *o, float *lse, void *ws, size_t ws_bytes,
                       void *stream)
{
    return run_fwd(p, false, SPARSE, nullptr, q, k, v, block_idx, o, lse, ws, ws_bytes, stream);
}

nsa_status nsa_sel_bwd(const nsa_problem *p, const void *q, const void *k, const void *v,
                       const void *o, const void *dO, const float *lse, const int32_t *block_idx,
                       void *dq, void *dk, void *dv, void *ws, size_t ws_bytes, void *stream)
{
    return run_bwd(p, false, SPARSE, nullptr, q, k, v, o, dO, lse, block_idx, nullptr, dq, dk, dv, ws,
                   ws_bytes, stream);
}

nsa_status nsa_dense_causal_fwd(const nsa_problem *p, const void *q, const void *k,
                                const void *v, void *o, float *lse, void *ws, size_t ws_bytes,
                                void *stream)
{
    return run_fwd(p, false, DENSE, nullptr, q, k, v, nullptr, o, lse, ws, ws_bytes, stream);
}

nsa_status nsa_dense_causal_bwd(const nsa_problem *p, const void *q, const void *k,
                                const void *v, const void *o, const void *dO, const float *lse,
                                void *dq, void *dk, void *dv, void *ws, size_t ws_bytes,
                                void *stream)
{
    return run_bwd(p, false, DENSE, nullptr, q, k, v, o, dO, lse, nullptr, nullptr, dq, dk, dv, ws,
                   ws_bytes, stream);
}

nsa_status nsa_sel_varlen_fwd(const nsa_problem *p, const int32_t *cu_seqlens, const void *q,
                              const void *k, const void *v, const int32_t *block_idx, void *o,
                              float *lse, void *ws, size_t ws_bytes, void *stream)
{
    return run_fwd(p, true, SPARSE, cu_seqlens, q, k, v, block_idx, o, lse, ws, ws_bytes, stream);
}

nsa_status nsa_sel_varlen_bwd(const nsa_problem *p, const int32_t *cu_seqlens, const void *q,
                              const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, const int32_t *block_idx, void *dq, void *dk,
                              void *dv, void *ws, size_t ws_bytes, void *stream)
{
    return run_bwd(p, true, SPARSE, cu_seqlens, q, k, v, o, dO, lse, block_idx, nullptr, dq, dk, dv, ws,
                   ws_bytes, stream);
}

size_t nsa_plan_size(const nsa_problem *p)
{
    Geo g;
    if (!p)
        return 0;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (make_geo(p, thd, SPARSE, thd ? (const int32_t *)16 : nullptr, g) != NSA_OK)
        return 0;
    return plan_layout(g, p->dtype).total;
}

size_t nsa_bwd_planned_workspace_size(const nsa_problem *p)
{
    Geo g;
    if (!p)
        return 0;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (make_geo(p, thd, SPARSE, thd ? (const int32_t *)16 : nullptr, g) != NSA_OK)
        return 0;
    return bwd_layout(g, p->dtype).plan;
}

nsa_status nsa_plan_build(const nsa_problem *p, const int32_t *cu_seqlens, const int32_t *block_idx, void *plan,
                          size_t plan_bytes, void *stream)
{
    Geo g;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    nsa_status s = make_geo(p, thd, SPARSE, cu_seqlens, g);
    if (s != NSA_OK)
        return s;
    if (!block_idx)
        return NSA_ERR_INVALID_ARG;
    const PlanLayout L = plan_layout(g, p->dtype);
    if ((s = check_ws(plan, plan_bytes, L.total)) != NSA_OK)
        return s;
    char *pl8 = (char *)plan;
    cudaStream_t st = (cudaStream_t)stream;
    if ((s = build_plan(g, block_idx, pl8, L, &((WsHeader *)pl8)->err, st)) != NSA_OK)
        return s;
    if (L.has_utable)  // the dQ kernel's query-tile unions, tiles grouped by shared blocks
        // over 128-token windows: a plan is built once, so the better grouping's time is paid once
        NSA_LAUNCH("qtile_unions", launch_qtile_unions(g, block_idx, (int *)(pl8 + L.utable), st, true, 4));
    return NSA_OK;
}

nsa_status nsa_sel_bwd_planned(const nsa_problem *p, const int32_t *cu_seqlens, const void *q, const void *k,
                               const void *v, const void *o, const void *dO, const float *lse,
                               const int32_t *block_idx, const void *plan, void *dq, void *dk, void *dv, void *ws,
                               size_t ws_bytes, void *stream)
{
    if (!p)
        return NSA_ERR_INVALID_ARG;
    if (!plan)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_bwd(p, thd, SPARSE, cu_seqlens, q, k, v, o, dO, lse, block_idx, plan, dq, dk, dv, ws, ws_bytes,
                   stream);
}

nsa_status nsa_swa_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const void *q,
                       const void *k, const void *v, void *o, float *lse, void *ws, size_t ws_bytes, void *stream)
{
    if (!p || window < 1)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_fwd(p, thd, DENSE, cu_seqlens, q, k, v, nullptr, o, lse, ws, ws_bytes, stream, window);
}

nsa_status nsa_swa_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const void *q,
                       const void *k, const void *v, const void *o, const void *dO, const float *lse, void *dq,
                       void *dk, void *dv, void *ws, size_t ws_bytes, void *stream)
{
    if (!p || window < 1)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_bwd(p, thd, DENSE, cu_seqlens, q, k, v, o, dO, lse, nullptr, nullptr, dq, dk, dv, ws, ws_bytes,
                   stream, window);
}

nsa_status nsa_sink_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const float *sinks,
                        const void *q, const void *k, const void *v, void *o, float *lse, void *ws,
                        size_t ws_bytes, void *stream)
{
    if (!p || window < 0 || !sinks || ((uintptr_t)sinks & 3))
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_fwd(p, thd, DENSE, cu_seqlens, q, k, v, nullptr, o, lse, ws, ws_bytes, stream, window, sinks);
}

nsa_status nsa_sink_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens, const float *sinks,
                        const void *q, const void *k, const void *v, const void *o, const void *dO,
                        const float *lse, void *dq, void *dk, void *dv, float *dsinks, void *ws,
                        size_t ws_bytes, void *stream)
{
    if (!p || window < 0 || !sinks || !dsinks || ((uintptr_t)sinks & 3) || ((uintptr_t)dsinks & 3))
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_bwd(p, thd, DENSE, cu_seqlens, q, k, v, o, dO, lse, nullptr, nullptr, dq, dk, dv, ws, ws_bytes,
                   stream, window, sinks, dsinks);
}

size_t nsa_causal_fwd_workspace_size(const nsa_problem *p) { return fwd_ws_need(p, CAUSAL); }

size_t nsa_causal_bwd_workspace_size(const nsa_problem *p) { return bwd_ws_need(p, CAUSAL); }

nsa_status nsa_causal_fwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, const void *q, const void *k, const void *v, void *o,
                          float *lse, void *ws, size_t ws_bytes, void *stream)
{
    if (!p || window < 0)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens_q != nullptr) || thd != (cu_seqlens_k != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_fwd(p, thd, CAUSAL, cu_seqlens_q, q, k, v, nullptr, o, lse, ws, ws_bytes, stream, window, nullptr,
                   cu_seqlens_k);
}

nsa_status nsa_causal_bwd(const nsa_problem *p, int32_t window, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, const void *q, const void *k, const void *v, const void *o,
                          const void *dO, const float *lse, void *dq, void *dk, void *dv, void *ws,
                          size_t ws_bytes, void *stream)
{
    if (!p || window < 0)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    if (thd != (cu_seqlens_q != nullptr) || thd != (cu_seqlens_k != nullptr))
        return NSA_ERR_INVALID_ARG;
    return run_bwd(p, thd, CAUSAL, cu_seqlens_q, q, k, v, o, dO, lse, nullptr, nullptr, dq, dk, dv, ws, ws_bytes,
                   stream, window, nullptr, nullptr, cu_seqlens_k);
}

nsa_status nsa_do_dot(const nsa_problem *p, const int32_t *cu_seqlens, const void *o,
                      const void *dO, float *delta, void *stream)
{
    Geo g;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    nsa_status s = make_geo(p, thd, DENSE, cu_seqlens, g);
    if (s != NSA_OK)
        return s;
    if (!o || !dO || !delta || !aligned16(o) || !aligned16(dO))
        return NSA_ERR_INVALID_ARG;
    if (g.ntok == 0)
        return NSA_OK;
    return cuda_status(launch_do_dot(g, o, dO, delta, p->dtype, (cudaStream_t)stream));
}

int64_t nsa_inverse_index_offsets_len(const nsa_problem *p)
{
    if (!p || p->block_size < 1 || p->T < 1)
        return 0;
    return (int64_t)p->B * p->Hkv * ((p->T + p->block_size - 1) / p->block_size) + 1;
}

nsa_status nsa_build_inverse_index(const nsa_problem *p, const int32_t *cu_seqlens,
                                   const int32_t *block_idx, int32_t *offsets, int32_t *rows,
                                   void *ws, size_t ws_bytes, void *stream)
{
    Geo g;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    nsa_status s = make_geo(p, thd, SPARSE, cu_seqlens, g);
    if (s != NSA_OK)
        return s;
    if (!block_idx || !offsets || !rows)
        return NSA_ERR_INVALID_ARG;
    if ((s = check_ws(ws, ws_bytes, nsa_bwd_workspace_size(p))) != NSA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    char *w8 = (char *)ws;
    WsHeader *hdr = (WsHeader *)ws;
    const PlanLayout L = plan_layout(g);
    NSA_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
    return build_csr(g, block_idx, (int *)(w8 + L.counts), offsets, rows, (Unit *)(w8 + L.units),
                     (int *)(w8 + L.nchunk), (int *)(w8 + L.slot), hdr, &hdr->err, L.chunk, st,
                     (int *)(w8 + L.chunkc));
}

nsa_status nsa_build_inverse_index_noalloc(const nsa_problem *p, const int32_t *cu_seqlens,
                                           const int32_t *block_idx, int32_t *offsets,
                                           int32_t *rows, int32_t *status_out, void *stream)
{
    Geo g;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    nsa_status s = make_geo(p, thd, SPARSE, cu_seqlens, g);
    if (s != NSA_OK)
        return s;
    if (!block_idx || !offsets || !rows || ((uintptr_t)status_out & 3))
        return NSA_ERR_INVALID_ARG;
    // scratch plan: header | counts | unit list | chunks per block | partial slots
    const PlanLayout L = plan_layout(g);
    const size_t nbgj = (size_t)g.B * g.Hkv * g.nbmax;
    const size_t off_counts = kAlign;
    const size_t off_units = align_up(off_counts + sizeof(int) * nbgj);
    const size_t off_nchunk = align_up(off_units + sizeof(Unit) * (size_t)L.max_units);
    const size_t off_slot = align_up(off_nchunk + sizeof(int) * nbgj);
    const size_t need = align_up(off_slot + sizeof(int) * nbgj);
    if (need > kNoallocScratchBytes)
        return NSA_ERR_UNSUPPORTED;
    void *base = nullptr;
    if ((s = noalloc_scratch_address(&base)) != NSA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    char *w8 = (char *)base;
    WsHeader *hdr = (WsHeader *)base;
    // the array keeps the previous call's contents: clear the error word here;
    // build_csr zeroes the per-block counts itself
    NSA_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
    if ((s = build_csr(g, block_idx, (int *)(w8 + off_counts), offsets, rows, (Unit *)(w8 + off_units),
                       (int *)(w8 + off_nchunk), (int *)(w8 + off_slot), hdr, &hdr->err, L.chunk, st)) != NSA_OK)
        return s;
    if (status_out)
        NSA_TRY(cudaMemcpyAsync(status_out, &hdr->err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    return NSA_OK;
}

nsa_status nsa_debug_stall(int32_t kernel, int32_t wait_limit_us)
{
    if (kernel < WAIT_TEST_NONE || kernel > WAIT_TEST_DQ || wait_limit_us < 0 || wait_limit_us > 2000000)
        return NSA_ERR_INVALID_ARG;
    g_wait_test.kernel = kernel;
    g_wait_test.wait_us = wait_limit_us;
    return NSA_OK;
}

nsa_status nsa_get_error(void *ws, void *stream, int32_t *out)
{
    if (!ws || !out)
        return NSA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return NSA_ERR_CUDA;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return NSA_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess)
        return NSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return NSA_ERR_CUDA;
    *out = v;
    return NSA_OK;
}

const char *nsa_status_string(int32_t s)
{
    switch (s) {
    case NSA_OK: return "NSA_OK";
    case NSA_ERR_INVALID_ARG: return "NSA_ERR_INVALID_ARG";
    case NSA_ERR_UNSUPPORTED: return "NSA_ERR_UNSUPPORTED";
    case NSA_ERR_BAD_INDEX: return "NSA_ERR_BAD_INDEX";
    case NSA_ERR_DEVICE_TIMEOUT: return "NSA_ERR_DEVICE_TIMEOUT";
    case NSA_ERR_CUDA: return "NSA_ERR_CUDA";
    case NSA_ERR_WORKSPACE: return "NSA_ERR_WORKSPACE";
    default: return "NSA_ERR_UNKNOWN";
    }
}

nsa_status nsa_trace_enable(int32_t max_records)
{
    if (g_trace) {
        for (int i = 0; i < g_trace_cap; ++i) {
            cudaEventDestroy(g_trace[i].start);
            cudaEventDestroy(g_trace[i].stop);
        }
        delete[] g_trace;
        g_trace = nullptr;
        g_trace_cap = g_trace_n = 0;
    }
    if (max_records <= 0)
        return NSA_OK;
    g_trace = new TraceRec[max_records];
    for (int i = 0; i < max_records; ++i) {
        g_trace[i].name = "";
        if (cudaEventCreate(&g_trace[i].start) != cudaSuccess || cudaEventCreate(&g_trace[i].stop) != cudaSuccess)
            return NSA_ERR_CUDA;
    }
    g_trace_cap = max_records;
    g_trace_n = 0;
    return NSA_OK;
}

void nsa_trace_reset(void) { g_trace_n = 0; }

int32_t nsa_trace_count(void) { return g_trace_n; }

nsa_status nsa_trace_get(int32_t i, const char **name, float *ms)
{
    if (!g_trace || i < 0 || i >= g_trace_n || !name || !ms)
        return NSA_ERR_INVALID_ARG;
    if (cudaEventSynchronize(g_trace[i].stop) != cudaSuccess)
        return NSA_ERR_CUDA;
    if (cudaEventElapsedTime(ms, g_trace[i].start, g_trace[i].stop) != cudaSuccess)
        return NSA_ERR_CUDA;
    *name = g_trace[i].name;
    return NSA_OK;
}

// ---- the step that produces the index (block selection) -------------------

size_t nsa_select_workspace_size(const nsa_problem *p)
{
    Geo g;
    const bool thd = p && p->layout == NSA_LAYOUT_THD;
    return select_geo(p, thd ? kFakeCuQ : nullptr, g, DENSE) == NSA_OK ? align_up(sizeof(WsHeader)) : 0;
}

nsa_status nsa_compress_keys_mean(const nsa_problem *p, const int32_t *cu_seqlens, const void *k, void *kc,
                                  void *stream)
{
    Geo g;
    nsa_status s = select_geo(p, cu_seqlens, g, DENSE);
    if (s != NSA_OK)
        return s;
    if (!k || !kc || !aligned16(k) || !aligned16(kc))
        return NSA_ERR_INVALID_ARG;
    if (g.ntok == 0 || g.nbmax == 0)
        return NSA_OK;
    cudaStream_t st = (cudaStream_t)stream;
    NSA_LAUNCH("compress_mean", launch_compress_mean(g, k, kc, p->dtype, st));
    return NSA_OK;
}

nsa_status nsa_block_scores(const nsa_problem *p, const int32_t *cu_seqlens, const void *q, const void *kc,
                            float *scores, void *ws, size_t ws_bytes, void *stream)
{
    Geo g;
    nsa_status s = select_geo(p, cu_seqlens, g, DENSE);
    if (s != NSA_OK)
        return s;
    if (!q || !kc || !scores || !aligned16(q) || !aligned16(kc) || ((uintptr_t)scores & 3u))
        return NSA_ERR_INVALID_ARG;
    if (!scores_gtc_supported(g, p->dtype))
        return NSA_ERR_UNSUPPORTED;
    if ((s = check_ws(ws, ws_bytes, align_up(sizeof(WsHeader)))) != NSA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    WsHeader *hdr = (WsHeader *)ws;
    NSA_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
    if (g.ntok == 0)
        return NSA_OK;
    NSA_LAUNCH("block_scores", launch_scores_gtc(g, q, kc, scores, p->dtype, &hdr->err, st));
    return NSA_OK;
}

nsa_status nsa_select_topk(const nsa_problem *p, const int32_t *cu_seqlens, const float *scores, int32_t *idx,
                           void *stream)
{
    Geo g;
    nsa_status s = select_geo(p, cu_seqlens, g, SPARSE);
    if (s != NSA_OK)
        return s;
    if (!scores || !idx || ((uintptr_t)scores & 3u) || ((uintptr_t)idx & 3u))
        return NSA_ERR_INVALID_ARG;
    if (g.ntok == 0)
        return NSA_OK;
    cudaStream_t st = (cudaStream_t)stream;
    NSA_LAUNCH("select_topk", launch_select_topk(g, scores, idx, st));
    return NSA_OK;
}

nsa_status nsa_count_pairs(const nsa_problem *p, const int32_t *cu_seqlens,
                           const int32_t *block_idx, int64_t *out_pairs, void *stream)
{
    Geo g;
    if (!p)
        return NSA_ERR_INVALID_ARG;
    const bool thd = p->layout == NSA_LAYOUT_THD;
    nsa_status s = make_geo(p, thd, SPARSE, cu_seqlens, g);
    if (s != NSA_OK)
        return s;
    if (!block_idx || !out_pairs)
        return NSA_ERR_INVALID_ARG;
    return cuda_status(launch_count_pairs(g, block_idx, (long long *)out_pairs, (cudaStream_t)stream));
}

}  // extern "C"
