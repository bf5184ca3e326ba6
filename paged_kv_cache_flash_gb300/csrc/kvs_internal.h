// Internal declarations shared by the host layer (kvs_host.cpp) and the CUDA
// translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kvs.h"

namespace kvs {

constexpr int kBlockTokens = 16;
constexpr int kChunkBlocks = 64;      // blocks per decode work item (split-K chunk)
constexpr int kMaxGroup = 8;          // query heads per KV head handled by one warp
constexpr int kStages = 4;            // TMA ring depth per warp
constexpr int kMaxCallSeqs = KVS_MAX_CALL_SEQS;

// Device error word bits (set by kernels, read by kvs_check_device).
enum : uint32_t {
    kErrBadPage = 1u << 0,       // block-table entry outside the pool
    kErrTmaTimeout = 1u << 1,    // an mbarrier wait ran out
    kErrBadRecord = 1u << 2,     // scoring met an inconsistent record
};

// One sequence of the current decode set, in call order.
struct DSeq {
    uint32_t slot;      // sequence slot (row of table / records / mass)
    uint32_t ntok;      // tokens (including the one appended for this step)
    uint32_t nb;        // blocks = ceil(ntok / 16)
    uint32_t blk_off;   // prefix of nb over call order (per-block LSE index)
    uint32_t item_off;  // prefix of CTA work items over call order
    uint32_t part_off;  // prefix of per-warp partials over call order
    uint32_t nchunk;    // ceil(nb / kChunkBlocks)
    uint32_t pad;
    uint64_t seq_id;
};

// The decode set, uploaded once per decode call (or debug_set_mass).
struct DSet {
    uint32_t nseq;
    uint32_t nb_total;
    uint32_t n_items;
    uint32_t n_parts;
    uint64_t t;                       // step counter after the decode
    uint32_t wg;                      // KV heads (warps) per work item
    uint32_t pad;
    DSeq seq[kMaxCallSeqs];
    uint32_t sorted[kMaxCallSeqs];    // call indices, ascending seq_id
    uint32_t srt_off[kMaxCallSeqs + 1];  // record-order prefix of nb over `sorted`
};

// Geometry and device pointers every kernel may need.
struct Geo {
    uint32_t L, Hq, Hkv, d, G;
    uint32_t pool_blocks, max_seqs, mb;  // mb = max_blocks_per_seq
    uint64_t page_bytes;
};

struct Work {             // carved out of the caller's workspace buffer
    uint32_t *err;        // error word
    uint32_t *err_info;   // first offending value
    uint32_t *counter;    // decode work counter (reset by the combine kernel)
    uint32_t *sel_count;  // selected records
    uint64_t *sel_thr;    // LOWFRAC threshold key: [0] prio bits, [1] record index
    DSet *dset;
    float2 *part_ml;      // [n_parts][8] (running max in log2 units, sum)
    float *part_o;        // [n_parts][8][d] unnormalised output
    float *lse_blk;       // [L*Hq][nb_total] per-block log2-sum-exp
    float *lse_head;      // [nseq][L*Hq] log2-sum-exp per head
    uint32_t *tile_cnt;   // [tiles] selection counts
    kvs_key *sel_ids;     // [nb_max] selected keys
    int32_t *sel_pages;   // [nb_max] page of each selected key
    uint32_t *sel_recidx; // [nb_max] record-order index of each selected key
    kvs_record *sel_recs; // [nb_max] record of each selected key
    uint8_t *ring;        // device side of the upload ring
};

struct Layout {           // byte offsets inside the workspace
    size_t err, counter, sel_count, sel_thr, dset, part_ml, part_o, lse_blk,
        lse_head, tile_cnt, sel_ids, sel_pages, sel_recidx, sel_recs, ring, total;
    size_t ring_slot_bytes;
    uint32_t ring_slots;
    uint32_t nb_max, parts_max, tiles_max;
};

Layout workspace_layout(const kvs_config &cfg);
Work carve(const Layout &lay, void *workspace);

// Entry in a page/record patch list (demote, readmit).
struct Patch {
    uint32_t slot;
    uint32_t block;
    int32_t page;         // new table entry (-1 = none)
    uint32_t has_record;  // 1: write `rec` into the record slot
    kvs_record rec;
};

// Append of n tokens to one sequence.
struct AppendArgs {
    const uint16_t *k, *v;     // [n][L][Hkv][d]
    uint16_t *pool;
    int32_t *table;
    kvs_record *records;
    const int32_t *pages;      // page of each touched block, from block first_blk
    uint32_t slot, p0, n;      // first token position, token count
    uint32_t first_blk, nblk;  // touched blocks
    uint32_t first_new;        // first block index that is new (>= first_blk)
    uint64_t seq_id, t_create;
};

// ---- launchers (each returns the cudaGetLastError() of its launch) -------
cudaError_t launch_append(const Geo &g, const AppendArgs &a, cudaStream_t s);
cudaError_t launch_decode(const Geo &g, const CUtensorMap &tmap, const Work &w,
                          const uint16_t *q, const int32_t *table,
                          uint32_t n_items, uint32_t wg, int grid, cudaStream_t s);
cudaError_t launch_combine(const Geo &g, const Work &w, float *out, uint32_t nseq,
                           cudaStream_t s);
cudaError_t launch_mass(const Geo &g, const Work &w, float *mass, uint32_t nb_total,
                        cudaStream_t s);
cudaError_t launch_score(const Geo &g, const Work &w, kvs_record *rec, const float *mass,
                         double alpha, uint32_t W, double wR, double wE, double wN,
                         double lo, double hi, uint32_t nb_total, cudaStream_t s);
cudaError_t launch_radix_select(const Geo &g, const Work &w, const kvs_record *rec,
                                uint32_t nb_total, uint32_t k, cudaStream_t s);
cudaError_t launch_select(const Geo &g, const Work &w, const kvs_record *rec,
                          const int32_t *table, int mode, uint32_t nb_total,
                          cudaStream_t s);
cudaError_t launch_gather(const Geo &g, const uint16_t *pool, const int32_t *pages,
                          uint32_t npages, uint8_t *staging, cudaStream_t s);
cudaError_t launch_patch(const Geo &g, int32_t *table, kvs_record *rec,
                         const Patch *p, uint32_t n, cudaStream_t s);
cudaError_t launch_copy_mass(const Geo &g, const Work &w, const float *src, float *mass,
                             uint32_t nseq, cudaStream_t s);

int decode_blocks_per_sm(const Geo &g, uint32_t wg);
size_t decode_smem_bytes(const Geo &g, uint32_t wg);

}  // namespace kvs
