// Kernel launchers, defined in the CUDA translation units and called by the
// host layer (kvs_host.cpp, kvs_noalloc.cu).  Not part of the public ABI.
#pragma once

#include "kvs_internal.h"

namespace kvs {

// ---- launchers (each returns the cudaGetLastError() of its launch) -------
// sa_dev: the entries in device memory; null -> taken from sa_host into the
// kernel's parameters (nseq <= kStepInline)
cudaError_t launch_append_step(const Geo &g, const uint16_t *k, const uint16_t *v, uint16_t *pool,
                               int32_t *table, kvs_record *records, uint8_t *page_clean,
                               const StepAppend *sa_dev, const StepAppend *sa_host, uint32_t nseq,
                               uint32_t rows_total, uint64_t t_create, cudaStream_t s);
cudaError_t launch_append(const Geo &g, const AppendArgs &a, cudaStream_t s);
cudaError_t launch_decode(const Geo &g, const CUtensorMap &tmap, const Work &w,
                          const uint16_t *q, const int32_t *table,
                          uint32_t n_items, uint32_t wg, int grid, cudaStream_t s);
cudaError_t launch_combine(const Geo &g, const Work &w, float *out, uint32_t nseq,
                           uint32_t max_nb, uint32_t max_nchunk, uint32_t sm_count, cudaStream_t s);
// Block masses into mass ([slot][mb]); with score != nullptr the kernel also
// scores every block of the set (records updated as by launch_score).
cudaError_t launch_mass(const Geo &g, const Work &w, float *mass, uint32_t nb_total, kvs_record *recs,
                        const ScoreArgs *score, cudaStream_t s);
cudaError_t launch_score(const Geo &g, const Work &w, kvs_record *rec, const float *mass,
                         double alpha, uint32_t W, double wR, double wE, double wN,
                         double lo, double hi, uint32_t nb_total, cudaStream_t s);
// alpha: the EMA weight (LRFU mode: the key's slope -ln(1 - alpha) is taken
// on the device, by the same fixed sequence of fp64 operations as the key)
cudaError_t launch_radix_select(const Geo &g, const Work &w, const kvs_record *rec,
                                uint32_t nb_total, uint32_t k, int mode, double alpha, cudaStream_t s);
cudaError_t launch_select(const Geo &g, const Work &w, const kvs_record *rec, const int32_t *table,
                          int mode, double alpha, uint32_t nb_total, bool count_pages, const SelectOut &out,
                          cudaStream_t s);
uint32_t select_launches(uint32_t nb_total);   // kernels launch_select issues
// Selection and gather plan in one kernel (launch_select + launch_plan), for
// sets of at most select_plan_fits records; out: ids (cap), slots, counts.
bool select_plan_fits(uint32_t nb_total);
cudaError_t launch_select_plan(const Geo &g, const Work &w, const kvs_record *rec, const int32_t *table, int mode,
                               double alpha, uint32_t nb_total, uint32_t mirror, const SelectOut &out,
                               cudaStream_t s);
cudaError_t launch_plan(const Work &w, uint32_t mirror, const SelectOut &out, cudaStream_t s);
cudaError_t launch_scatter(const Geo &g, const uint8_t *staging, const int32_t *pages, uint32_t npages,
                           uint16_t *pool, cudaStream_t s);
// hdr_dev: pinned, mapped words [0..4] that receive the counts and then seq
// once the copies are visible to the host (null: no completion word)
cudaError_t launch_mirror_copy(const Geo &g, const Work &w, const uint16_t *pool, void *host_dev,
                               uint32_t pool_blocks, int grid, uint32_t *hdr_dev, uint32_t seq, cudaStream_t s);
cudaError_t launch_gather(const Geo &g, const uint16_t *pool, const int32_t *pages,
                          uint32_t npages, uint8_t *staging, cudaStream_t s);
// bytes (<= kSetInlineBytes) from host memory src to device memory dst, in
// a kernel's parameters (no copy engine operation)
cudaError_t launch_set(const void *src, size_t bytes, void *dst, cudaStream_t s);
cudaError_t launch_patch(const Geo &g, int32_t *table, kvs_record *rec, uint8_t *page_clean,
                         const Patch *p, uint32_t n, cudaStream_t s);
cudaError_t launch_kivi_compress(const Geo &g, const KiviJob *jobs, uint32_t njobs, const uint8_t *pool,
                                 uint8_t *gpool, int32_t *table, cudaStream_t s);
cudaError_t launch_decode_kivi(const Geo &g, const Work &w, const uint16_t *q, const int32_t *table,
                               const uint8_t *gpool, uint32_t n_items, int grid, cudaStream_t s);
int decode_kivi_blocks_per_sm(const Geo &g);
cudaError_t launch_prefetch_plan(const PrefCand *cand, uint32_t n, uint32_t k, uint64_t *keys,
                                 uint64_t *out_key, uint32_t *out_idx, cudaStream_t s);
cudaError_t launch_copy_mass(const Geo &g, const Work &w, const float *src, float *mass,
                             uint32_t nseq, cudaStream_t s);

int decode_blocks_per_sm(const Geo &g, uint32_t wg);
size_t decode_smem_bytes(const Geo &g, uint32_t wg);

}  // namespace kvs
