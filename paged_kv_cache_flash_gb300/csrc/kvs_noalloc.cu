// kvs_decode_noalloc: decode attention and per-block mass for one sequence,
// for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// allocate anything else on the GPU: code that runs inside a host program's
// own memory budget or allocator (a plugin or custom operator of another
// framework), or a serving loop that forbids allocation after start-up so
// that latency and memory use stay fixed.  Such a caller cannot provide the
// decode kernel's scratch (chunk partials and per-block log-sum-exp), so this
// entry point keeps that scratch in one fixed array compiled into the
// library, below.  Every GPU that loads the library holds the array until the
// process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  What must start at zero (the work counter and the error word)
// is cleared at the start of each call; the rest is fully written before it
// is read.  Two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array: order them.
//
// The kernels' error word (a block-table entry outside the pool, replaced by
// page 0 before any access; a TMA wait that ran out) lives in the array too;
// a caller that passes `status` gets it, with the first offending value,
// copied there in stream order after the outputs.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "kvs_internal.h"
#include "kvs_launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(48) << 20;   // 48 MiB per GPU

__device__ __align__(256) static uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_dev[kMaxDevices];      // device address of the array, per device
int g_sm_count[kMaxDevices];
int g_per_sm[kMaxDevices][2][3];       // occupancy per (d = 64/128, wg = 1/2/4)

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int say(char *msg, size_t n, int code, const char *text)
{
    if (msg && n) {
        std::strncpy(msg, text, n - 1);
        msg[n - 1] = 0;
    }
    return code;
}

}  // namespace

extern "C" int kvs_decode_noalloc(uint32_t num_layers, uint32_t num_q_heads, uint32_t num_kv_heads,
                                  uint32_t head_dim, const void *pool, uint32_t pool_blocks,
                                  const int32_t *block_table, uint32_t n_tokens, const void *q,
                                  float *out, float *mass, uint32_t *status, void *stream, char *msg,
                                  size_t msg_bytes)
{
    using namespace kvs;
    char buf[256];
    if (!pool || !block_table || !q || !out || !mass)
        return say(msg, msg_bytes, KVS_EINVAL, "pool, block_table, q, out and mass must be given");
    if (head_dim != 64 && head_dim != 128)
        return say(msg, msg_bytes, KVS_EINVAL, "head_dim must be 64 or 128");
    if (!num_layers || !num_kv_heads || !num_q_heads || num_q_heads % num_kv_heads ||
        num_q_heads / num_kv_heads > static_cast<uint32_t>(kMaxGroup))
        return say(msg, msg_bytes, KVS_EINVAL, "head counts: Hq a multiple of Hkv, at most 8 per KV head");
    if (!n_tokens || !pool_blocks || static_cast<uint64_t>(num_layers) * pool_blocks >= (1ull << 31))
        return say(msg, msg_bytes, KVS_EINVAL, "n_tokens and pool_blocks must be > 0 (layers*pool_blocks < 2^31)");
    if ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(q) |
         reinterpret_cast<uintptr_t>(out)) % 16)
        return say(msg, msg_bytes, KVS_EINVAL, "pool, q and out must be 16-byte aligned");

    Geo g{};
    g.L = num_layers;
    g.Hq = num_q_heads;
    g.Hkv = num_kv_heads;
    g.d = head_dim;
    g.G = num_q_heads / num_kv_heads;
    g.pool_blocks = pool_blocks;
    g.max_seqs = 1;
    const uint32_t nb = (n_tokens + kBlockTokens - 1) / kBlockTokens;
    g.mb = nb;
    g.page_bytes = static_cast<uint64_t>(2) * g.L * g.Hkv * kBlockTokens * g.d * 2;
    g.fp8 = 0;            // bf16 pages only
    g.k_scale = g.v_scale = 1.f;
    const uint32_t wg = g.Hkv % 4 == 0 ? 4 : (g.Hkv % 2 == 0 ? 2 : 1);
    const uint32_t chunk = 64;
    const uint32_t nchunk = (nb + chunk - 1) / chunk;
    const size_t LH = static_cast<size_t>(g.L) * g.Hq;
    const size_t parts = static_cast<size_t>(g.L) * g.Hkv * nchunk;

    // scratch carved from the fixed array
    size_t o = 0;
    const size_t off_hdr = o;   o = up256(o + 256);
    const size_t off_set = o;   o = up256(o + sizeof(DSet));
    const size_t off_ml = o;    o = up256(o + parts * kMaxGroup * sizeof(float2));
    const size_t off_po = o;    o = up256(o + parts * kMaxGroup * g.d * sizeof(float));
    const size_t off_lb = o;    o = up256(o + LH * nb * sizeof(float));
    const size_t off_sm = o;    o = up256(o + static_cast<size_t>(g.L) * g.Hkv * nb * sizeof(float));
    if (o > kScratchBytes) {
        std::snprintf(buf, sizeof buf,
                      "this call needs %zu bytes of scratch; the built-in maximum is %zu bytes "
                      "(48 MiB): use kvs_decode_step with caller-provided workspace",
                      o, kScratchBytes);
        return say(msg, msg_bytes, KVS_EINVAL, buf);
    }

    // once per device, with that device current: the array's device address
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return say(msg, msg_bytes, KVS_ECUDA, "no usable current device");
    uint8_t *base;
    int grid_per_sm, sm_count;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_dev[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                std::snprintf(buf, sizeof buf, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
                return say(msg, msg_bytes, KVS_ECUDA, buf);
            }
            e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return say(msg, msg_bytes, KVS_ECUDA, "cannot read the SM count");
            g_scratch_dev[dev] = p;
        }
        int &per = g_per_sm[dev][g.d == 128][wg == 4 ? 2 : wg - 1];
        if (per == 0)
            per = decode_blocks_per_sm(g, wg);
        if (per < 1)
            return say(msg, msg_bytes, KVS_ECUDA, "decode kernel does not fit on an SM");
        base = static_cast<uint8_t *>(g_scratch_dev[dev]);
        grid_per_sm = per * g_sm_count[dev];
        sm_count = g_sm_count[dev];
    }

    Work w{};
    w.err = reinterpret_cast<uint32_t *>(base + off_hdr);
    w.err_info = w.err + 1;
    w.counter = w.err + 16;
    w.dset = reinterpret_cast<DSet *>(base + off_set);
    w.part_ml = reinterpret_cast<float2 *>(base + off_ml);
    w.part_o = reinterpret_cast<float *>(base + off_po);
    w.lse_blk = reinterpret_cast<float *>(base + off_lb);
    w.stream_mass = reinterpret_cast<float *>(base + off_sm);

    // the one-sequence decode set: header and one entry, sent in a kernel's
    // parameters (no copy-engine operation, no host buffer to keep alive)
    alignas(16) uint8_t set_bytes[kSetInlineBytes];
    static_assert(offsetof(DSet, seq) + sizeof(DSeq) <= kSetInlineBytes, "one-entry set fits the parameters");
    std::memset(set_bytes, 0, sizeof set_bytes);
    DSet &ds = *reinterpret_cast<DSet *>(set_bytes);
    ds.nseq = 1;
    ds.nb_total = nb;
    ds.n_items = g.L * g.Hkv * nchunk;
    ds.n_parts = static_cast<uint32_t>(parts);
    ds.wg = wg;
    ds.chunk = chunk;
    ds.chunk_big = chunk;       // uniform chunks: every chunk "big", the last one short
    ds.chunk_small = chunk;
    ds.seq[0].nbig = nchunk;
    ds.seq[0].ntok = n_tokens;
    ds.seq[0].nb = nb;
    ds.seq[0].nchunk = nchunk;
    ds.seq[0].srt_ci = 0;       // record order: the one sequence, from block 0
    ds.seq[0].srt_off = 0;

    // TMA descriptor of the caller's pool (host-side encoding only)
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaDriverEntryPointQueryResult qres;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void **>(&encode),
                                         12000, cudaEnableDefault, &qres);
    if (e != cudaSuccess || qres != cudaDriverEntryPointSuccess || !encode)
        return say(msg, msg_bytes, KVS_ECUDA, "cuTensorMapEncodeTiled not available");
    alignas(64) CUtensorMap tmap;
    const cuuint64_t d = g.d;
    cuuint64_t dims[5] = {d, kBlockTokens, g.Hkv, 2, static_cast<cuuint64_t>(g.L) * pool_blocks};
    cuuint64_t strides[4] = {d * 2, kBlockTokens * d * 2, g.Hkv * kBlockTokens * d * 2,
                             2ull * g.Hkv * kBlockTokens * d * 2};
    cuuint32_t box[5] = {64, kBlockTokens, 1, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return say(msg, msg_bytes, KVS_EINVAL, "pool cannot be described for TMA");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define NA_CHECK(call)                                                        \
    do {                                                                      \
        cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess) {                                              \
            std::snprintf(buf, sizeof buf, "%s: %s", #call, cudaGetErrorString(e_)); \
            return say(msg, msg_bytes, KVS_ECUDA, buf);                       \
        }                                                                     \
    } while (0)
    NA_CHECK(cudaMemsetAsync(base + off_hdr, 0, 256, s));
    NA_CHECK(launch_set(&ds, dset_bytes(1), w.dset, s));
    const int grid = static_cast<int>(std::min<uint32_t>((ds.n_items + wg - 1) / wg,
                                                         static_cast<uint32_t>(grid_per_sm)));
    NA_CHECK(launch_decode(g, tmap, w, static_cast<const uint16_t *>(q), block_table, ds.n_items, wg,
                           grid, s));
    NA_CHECK(launch_combine(g, w, out, 1, nb, nchunk, static_cast<uint32_t>(sm_count), s));
    NA_CHECK(launch_mass(g, w, mass, nb, nullptr, nullptr, s));
    if (status)     // error word and its first offending value, after the outputs
        NA_CHECK(cudaMemcpyAsync(status, w.err, 2 * sizeof(uint32_t), cudaMemcpyDeviceToDevice, s));
#undef NA_CHECK
    return KVS_OK;
}
