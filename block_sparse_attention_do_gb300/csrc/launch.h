// launch.h -- host-side launchers of the kernels, called by nsa_api.cu.
// Every launcher enqueues on `st` and returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>

#include "nsa_common.cuh"

namespace nsa {

// Self-test of the tensor-core kernels' bounded waits (nsa_debug_stall): the
// kernel whose S-product issuer stays idle, so that its first wait on S runs
// out, and the wait limit of every tensor-core kernel in microseconds
// (0: the default).  Both 0 in normal operation.
enum { WAIT_TEST_NONE = 0, WAIT_TEST_FWD = 1, WAIT_TEST_DKDV = 2, WAIT_TEST_DQ = 3 };
struct WaitTest {
    int kernel, wait_us;
};
WaitTest wait_test();

// ---- prep (k_prep.cu) ----------------------------------------------------
cudaError_t launch_do_dot(const Geo &g, const void *o, const void *dO, float *delta, int dtype,
                          cudaStream_t st);
cudaError_t launch_validate_index(const Geo &g, const int *idx, int *err, cudaStream_t st);
// counts[B*Hkv*nbmax] must be zeroed by the caller
cudaError_t launch_csr_count(const Geo &g, const int *idx, int *counts, int *err, cudaStream_t st);
// offsets (B*Hkv*nbmax + 1), units, per-block chunk table; chunk = tokens per unit
cudaError_t launch_csr_scan(const Geo &g, const int *counts, int *offsets, Unit *units,
                            int *blk_nchunk, int *blk_slot, WsHeader *hdr, int chunk,
                            cudaStream_t st);
cudaError_t launch_csr_fill(const Geo &g, const int *idx, const int *offsets, int *rows,
                            cudaStream_t st);
// the same inverse index by 32-token chunks: per-chunk histograms
// (chunk_counts, B*Hkv*nbmax*csr_nchunks(g) ints, turned into per-chunk
// prefixes in place; counts = list lengths), then an ordered per-chunk fill
int csr_nchunks(const Geo &g);
bool csr_chunked_ok(const Geo &g);
// delta = rowsum(dO * O) riding along the chunk count (see below)
struct DotArgs {
    const void *o, *dO;
    float *delta;
    int dtype;
};
// dot (nullable): also computes delta in the same launch
cudaError_t launch_csr_chunk_count(const Geo &g, const int *idx, int *chunk_counts, int *counts, int *err,
                                   cudaStream_t st, const DotArgs *dot = nullptr);
cudaError_t launch_csr_chunk_fill(const Geo &g, const int *idx, const int *chunk_prefix, const int *offsets,
                                  int *rows, cudaStream_t st);
// sums the fp32 partials of split blocks into dk/dv and zeroes unselected blocks
cudaError_t launch_dkdv_reduce(const Geo &g, const int *blk_nchunk, const int *blk_slot,
                               const float *partials, void *dk, void *dv, int dtype,
                               cudaStream_t st, bool dependent = false);
cudaError_t launch_count_pairs(const Geo &g, const int *idx, long long *out, cudaStream_t st);
// attention sinks: fold sinks[h] into the forward's o and lse in place; and
// dsinks[h] = -sum over head h's rows of exp(sinks[h] - lse) * delta
cudaError_t launch_sink_fwd(const Geo &g, const float *sinks, void *o, float *lse, int dtype, cudaStream_t st);
cudaError_t launch_sink_bwd(const Geo &g, const float *sinks, const float *lse, const float *delta, float *dsinks,
                            cudaStream_t st);

// ---- SIMT kernels (k_simt.cu): any supported shape, fp32 or bf16 ----------
cudaError_t launch_fwd_simt(const Geo &g, const void *q, const void *k, const void *v,
                            const int *idx, void *o, float *lse, int dtype, cudaStream_t st);
cudaError_t launch_dq_simt(const Geo &g, const void *q, const void *k, const void *v,
                           const void *dO, const float *lse, const float *delta, const int *idx,
                           void *dq, int dtype, cudaStream_t st);
cudaError_t launch_dkdv_simt(const Geo &g, const void *q, const void *k, const void *v,
                             const void *dO, const float *lse, const float *delta,
                             const int *offsets, const int *rows, void *dk, void *dv, int dtype,
                             cudaStream_t st);

// ---- tensor-core kernels for the other shapes (k_gtc.cu): bf16 with D in
// {32, 64, 128} and block_size in {16, 32, 64}, fp32 (split precision) with D
// in {32, 64}; one CTA per query tile or dK/dV unit ----------------------------
bool gtc_supported(const Geo &g, int dtype);
cudaError_t launch_fwd_gtc(const Geo &g, const void *q, const void *k, const void *v, const int *idx, void *o,
                           float *lse, int dtype, int *err, cudaStream_t st);
cudaError_t launch_dq_gtc(const Geo &g, const void *q, const void *k, const void *v, const void *dO,
                          const float *lse, const float *delta, const int *idx, void *dq, int dtype, int *err,
                          cudaStream_t st);
// max_units CTAs; those past the plan's unit count return at once
cudaError_t launch_dkdv_gtc(const Geo &g, const void *q, const void *k, const void *v, const void *dO,
                            const float *lse, const float *delta, const int *offsets, const int *rows,
                            const Unit *units, const WsHeader *hdr, int max_units, float *partials, void *dk,
                            void *dv, int dtype, int *err, cudaStream_t st);

// the selection step's block scores on the tensor cores (bf16, or fp32 by
// split precision; D in {32, 64, 128}); kc [B, Hkv, nbmax, D] dense
bool scores_gtc_supported(const Geo &g, int dtype);
cudaError_t launch_scores_gtc(const Geo &g, const void *q, const void *kc, float *scores, int dtype, int *err,
                              cudaStream_t st);

// ---- the selection step's other kernels (k_select.cu) ---------------------
// kc [B, Hkv, nbmax, D] dense: the mean of each complete block's keys, zero rows elsewhere
cudaError_t launch_compress_mean(const Geo &g, const void *k, void *kc, int dtype, cudaStream_t st);
// idx rows from block scores (rows as the index's; nbmax scores each)
cudaError_t launch_select_topk(const Geo &g, const float *scores, int *idx, cudaStream_t st);

// ---- tensor-core kernels (bf16, D = 128, block_size = 64) -----------------
bool tc_supported(const Geo &g, int dtype);
// tile_next: a device int that is zero when the kernel starts (its work counter).
// utable: the query-tile union table (launch_qtile_unions), or null (the kernel
// builds the unions); after_kernel: the launch directly follows a kernel of
// this library (the index validation or the union build) and becomes its
// programmatic dependent (it waits for it before reading utable)
cudaError_t launch_fwd_tc(const Geo &g, const void *q, const void *k, const void *v,
                          const int *idx, const int *utable, bool grouped, void *o, float *lse, int *err,
                          int *tile_next, bool after_kernel, cudaStream_t st);
// every query tile's block union for the dQ kernel, into utable
// (qtile_union_table_bytes(g) bytes; 0, and no launch, for the dense entries,
// whose unions are block ranges the dQ kernel builds itself); a
// programmatic dependent of the kernel before it on st
size_t qtile_union_table_bytes(const Geo &g);
// whether the table's tiles are grouped by shared blocks rather than made of
// consecutive tokens (qtile_group_kernel)
bool qtile_groupable(const Geo &g);
// group: tiles grouped by shared blocks where qtile_groupable, else
// consecutive tokens; tpl: tokens per lane of the grouping warp (2, 3 or 4:
// windows of 64, 96 or 128 tokens; a wider window groups better and takes
// longer)
cudaError_t launch_qtile_unions(const Geo &g, const int *idx, int *utable, cudaStream_t st, bool group,
                                int tpl = 2);
// utable: the union table launch_qtile_unions wrote, or null (dense
// entries); grouped: its tiles are grouped by shared blocks
cudaError_t launch_dq_tc(const Geo &g, const void *q, const void *k, const void *v,
                         const void *dO, const float *lse, const float *delta, const int *idx,
                         const int *utable, bool grouped, void *dq, int *err, int *tile_next, cudaStream_t st);
cudaError_t launch_dkdv_tc(const Geo &g, const void *q, const void *k, const void *v,
                           const void *dO, const float *lse, const float *delta,
                           const int *offsets, const int *rows, const Unit *units,
                           const WsHeader *hdr, int max_units, float *partials, void *dk, void *dv,
                           int *err, cudaStream_t st);

}  // namespace nsa
