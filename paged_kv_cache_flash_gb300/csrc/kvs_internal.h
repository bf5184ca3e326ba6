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
constexpr uint32_t kMaxChunk = 128;   // blocks per decode work item (split-K chunk): at most
constexpr uint32_t kMinChunk = 16;    //   ... and at least
constexpr int kMaxGroup = 8;          // query heads per KV head handled by one warp
constexpr int kStages = 6;            // mbarriers reserved per warp (rings use 3 (bf16) or 4 (FP8))
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
    uint32_t nchunk;    // chunks (work items per (layer, KV head)): nchunk_q + page chunks
    uint32_t nbig;      // page chunks of chunk_big blocks; the rest are of chunk_small
    uint32_t qb;        // KIVI: leading blocks held in 2-bit group pages (even), else 0
    uint32_t nchunk_q;  // KIVI: chunks over those blocks (partials 0 .. nchunk_q-1), else 0
    uint32_t nbig_q;    // KIVI: group-page chunks of `chunk` blocks; the rest of chunk_q_small
    uint32_t item_off_q;  // KIVI: prefix of group-page work items over call order
    // record order (ascending seq_id) -- these two describe the sequence at
    // POSITION i of that order, not the sequence of this entry:
    uint32_t srt_ci;      // its call index
    uint32_t srt_off;     // prefix of nb over the positions before it
    uint64_t seq_id;
};

// The decode set, uploaded once per decode call (or debug_set_mass).  The
// entries come last, so that a call uploads only the header and its nseq
// entries (dset_bytes).
struct DSet {
    uint32_t nseq;
    uint32_t nb_total;
    uint32_t n_items;                 // bf16 (or FP8) page items
    uint32_t n_items_q;               // KIVI group-page items
    uint32_t n_parts;
    uint64_t t;                       // step counter after the decode
    uint32_t wg;                      // KV heads (warps) per work item
    uint32_t chunk;                   // blocks per 2-bit group-page work item: the first nbig_q
    uint32_t chunk_q_small;           //   ... and the rest of each stream
    uint32_t chunk_big;               // blocks per page work item: the first nbig chunks
    uint32_t chunk_small;             //   ... and the rest of each stream
    DSeq seq[kMaxCallSeqs];
};

inline size_t dset_bytes(uint32_t nseq)
{
    return offsetof(DSet, seq) + static_cast<size_t>(nseq) * sizeof(DSeq);
}

// A decode set of at most this many bytes travels in a kernel's parameters
// (no upload copy).
constexpr size_t kSetInlineBytes = 4096;

// Parameters of the per-block scoring ("KV-Cache Offloading for LLM
// Inference -- Visual Reference" s.11-12): EMA weight, priority weights,
// tier cuts, recency window.
struct ScoreArgs {
    double alpha, wR, wE, wN, lo, hi;
    uint32_t W;
};

// Geometry and device pointers every kernel may need.
struct Geo {
    uint32_t L, Hq, Hkv, d, G;
    uint32_t pool_blocks, max_seqs, mb;  // mb = max_blocks_per_seq
    uint64_t page_bytes;
    uint32_t fp8;                        // pages hold E4M3 codes (1 byte per element)
    float k_scale, v_scale;              // FP8: value = code * scale
    uint32_t kivi;                       // 2-bit group pages behind a bf16 residual window
    uint32_t kivi_groups;                // group pages in the group pool
    uint64_t group_page_bytes;           // L * Hkv * KVS_KIVI_TILE_BYTES
};

struct Work {             // carved out of the caller's workspace buffer
    uint32_t *err;        // error word
    uint32_t *err_info;   // first offending value
    uint32_t *counter;    // decode work counters: [0] page items, [1] group-page items
                          // (reset by the combine kernel)
    uint32_t *sel_count;  // selected records
    uint64_t *sel_thr;    // LOWFRAC threshold key: [0] prio bits, [1] record index
    DSet *dset;
    float2 *part_ml;      // [n_parts][8] (running max in log2 units, sum)
    float *part_o;        // [n_parts][8][d] unnormalised output
    float *lse_blk;       // [L*Hq][nb_total] per-block log2-sum-exp
    float *stream_mass;   // [L*Hkv][nb_total] block mass of each (layer, KV head) stream
    uint32_t *tile_cnt;   // [tiles] selection counts
    kvs_key *sel_ids;     // [nb_max] selected keys
    int32_t *sel_pages;   // [nb_max] page of each selected key
    uint32_t *sel_recidx; // [nb_max] record-order index of each selected key
    kvs_record *sel_recs; // [nb_max] record of each selected key
    uint8_t *sel_full;    // [nb_max] 1 if the selected key's block holds 16 tokens
    uint32_t *dev_refcnt; // [pool_blocks] references per page (host-maintained mirror)
    uint32_t *page_cnt;   // [pool_blocks] selected references (zero between calls)
    uint32_t *page_first; // [pool_blocks] first selected position (~0 between calls)
    int32_t *page_pos;    // [pool_blocks] position of a page in the gather plan
    uint8_t *page_clean;  // [pool_blocks] 1: the host mirror holds the page's bytes
    int32_t *plan_pages;  // [nb_max] eligible pages, first-occurrence order
    int32_t *plan_slot;   // [nb_max] per selected key: host page index, -1 if none
    uint32_t *readback;   // [4 + nb_max]: n_selected, n_pages, n_copy, -, copy list
    uint8_t *ring;        // device side of the upload ring
};

// Optional direct outputs of a selection (null / 0 when unused): the caller's
// key and slot lists (their first ids_cap entries), and a host buffer, through
// its device mapping, for the counts (select_scatter_kernel writes one word,
// the selected count; plan_kernel four: selected, pages, pages copied, 0).
struct SelectOut {
    kvs_key *ids;
    int32_t *slots;
    uint32_t ids_cap;
    uint32_t *count_host;
};

struct Layout {           // byte offsets inside the workspace
    size_t err, counter, sel_count, sel_thr, dset, part_ml, part_o, lse_blk,
        stream_mass, tile_cnt, sel_ids, sel_pages, sel_recidx, sel_recs, sel_full, dev_refcnt,
        page_cnt, page_first, page_pos, page_clean, plan_pages, plan_slot, readback, ring, total;
    size_t ring_slot_bytes;
    uint32_t ring_slots;
    uint32_t nb_max, parts_max, tiles_max;
};

// One 32-token group of one sequence to quantise into a group page.
struct KiviJob {
    uint32_t slot;      // sequence slot (table row)
    uint32_t group;     // group index: blocks 2*group, 2*group+1
    int32_t page0, page1;  // bf16 pages of the two blocks
    uint32_t gpage;     // destination group page
    uint32_t pad;
};

// One demoted block as the prefetch plan sees it.
struct PrefCand {
    double ema;         // EMA score kept in the block's record
    uint32_t ntok;      // tokens of its sequence
    uint32_t block;     // block index
};
static_assert(sizeof(PrefCand) == 16, "PrefCand is 16 bytes");

Layout workspace_layout(const kvs_config &cfg);
Work carve(const Layout &lay, void *workspace);

// Entry in a page/record patch list (demote, readmit).
struct Patch {
    uint32_t slot;
    uint32_t block;
    int32_t page;         // new table entry (-1 = none)
    uint32_t what;        // kPatchRecord | kPatchPageWritten
    kvs_record rec;
};
enum : uint32_t {
    kPatchRecord = 1u,      // write `rec` into the record slot
    kPatchPageWritten = 2u, // the page's bytes were rewritten: host mirror is stale
};

// Append of n tokens to one sequence.
struct AppendArgs {
    const uint16_t *k, *v;     // [n][L][Hkv][d]
    uint16_t *pool;
    uint8_t *page_clean;       // cleared for every page written
    int32_t *table;
    kvs_record *records;
    const int32_t *pages;      // page of each touched block, from block first_blk
    uint32_t slot, p0, n;      // first token position, token count
    uint32_t first_blk, nblk;  // touched blocks
    uint32_t first_new;        // first block index that is new (>= first_blk)
    uint64_t seq_id, t_create;
};

// One sequence of a batched one-token append.
struct StepAppend {
    uint32_t slot;        // sequence slot
    uint32_t pos;         // token position (block = pos / 16)
    int32_t page;         // page of that block
    uint32_t nslots;      // slots written: 1, or 16 - pos % 16 when the token opens the block
    uint32_t row_off;     // prefix of nslots * L * 2 * Hkv over the call
    uint32_t fresh;       // 1: the block is new (record + table entry written)
    uint64_t seq_id;
};

// A step append of at most kStepInline sequences travels in the kernel's
// parameters (no upload copy ahead of the kernel).
constexpr uint32_t kStepInline = 16;
struct StepAppendInline {
    StepAppend e[kStepInline];
};

// Work items of one call (page items, and separately the 2-bit group-page
// items of a KIVI context).  Each (layer, KV head) stream of n blocks is
// cut into nbig(n) chunks of `big` blocks followed by chunks of `small`
// blocks over its last blocks (at least `tail` of them), and a sequence's
// items are claimed chunk by chunk (every stream's chunk 0, then chunk 1, ...):
// the small chunks come last, so that when the large ones run out every warp
// still finds short work and the launch ends evenly.  `tail` makes the small
// chunks of all streams at least half a large chunk per warp: when the large
// items run out, a warp has on average half of one left, so that much short
// work per warp evens the finish (a larger tail only adds partials and items).
struct PageChunks {
    uint32_t big, small, tail;
    uint32_t nbig(uint32_t n) const { return n > tail ? (n - tail) / big : 0; }
    uint32_t nchunk(uint32_t n) const
    {
        const uint32_t nb = nbig(n);
        return nb + (n - nb * big + small - 1) / small;
    }
};

// The largest big chunk (128, 64, 32, 16) whose large items alone give every
// one of the `workers` warps one to start with; small chunks of 16 blocks
// (or 32, 64, ... when the partials of 16 would not fit parts_cap with
// extra_parts).  If no big chunk gives every warp a large item, the smallest
// that fits.  big = 0 if nothing fits.
inline PageChunks pick_page_chunks(const uint32_t *nres, uint32_t n, uint32_t L, uint32_t Hkv,
                                   uint32_t workers, uint64_t parts_cap, uint64_t extra_parts)
{
    PageChunks best{0, 0, 0};
    const uint64_t streams = static_cast<uint64_t>(n) * L * Hkv;
    for (uint32_t c = kMaxChunk; c >= kMinChunk; c >>= 1) {
        bool fits = false;
        uint64_t big_items = 0;
        for (uint32_t sm = kMinChunk; sm <= c && !fits; sm <<= 1) {
            PageChunks pc;
            pc.big = c;
            pc.small = sm;
            const uint64_t t = (static_cast<uint64_t>(workers) * c / 2 + streams - 1) / streams;
            pc.tail = static_cast<uint32_t>((t + sm - 1) / sm * sm);
            uint64_t parts = extra_parts;
            big_items = 0;
            for (uint32_t i = 0; i < n; ++i) {
                parts += static_cast<uint64_t>(L) * Hkv * pc.nchunk(nres[i]);
                big_items += static_cast<uint64_t>(L) * Hkv * pc.nbig(nres[i]);
            }
            if (parts <= parts_cap) {
                fits = true;
                best = pc;
            }
        }
        if (!fits || big_items >= workers)
            break;
    }
    return best;
}

}  // namespace kvs
