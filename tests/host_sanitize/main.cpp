// Drives the host layer (kvs_host.cpp) through the calls that need no GPU,
// built with AddressSanitizer and UndefinedBehaviorSanitizer: configuration
// checks over valid and invalid configurations of every page format, the
// buffer sizes, the decode work-item plan over 300 seeded calls, failure
// injection, and context creation that fails before any device work (and
// must free everything it took).  Exits 0 when every expectation holds; the
// sanitizers abort the program on any memory or undefined-behaviour error.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "kvs.h"

namespace {

int failures = 0;

void expect(bool ok, const char *what)
{
    if (!ok) {
        std::fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

kvs_config base70b()
{
    kvs_config c;
    std::memset(&c, 0, sizeof c);
    c.num_layers = 80;
    c.num_q_heads = 64;
    c.num_kv_heads = 8;
    c.head_dim = 128;
    c.block_tokens = KVS_BLOCK_TOKENS;
    c.pool_blocks = 8200;
    c.max_seqs = 1;
    c.max_blocks_per_seq = 8197;
    c.staging_pages = 32;
    c.alpha = 0.15;
    c.recency_window = 64;
    c.w_recency = 0.25;
    c.w_ema = 0.55;
    c.w_anchor = 0.20;
    c.cut_lo = 0.3;
    c.cut_hi = 0.6;
    c.k_scale = c.v_scale = 1.0f;
    return c;
}

// splitmix64: seeded sizes for the plan calls
uint64_t mix(uint64_t &s)
{
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void sizes()
{
    kvs_sizes sz;
    kvs_config c = base70b();
    expect(kvs_required_sizes(&c, &sz) == KVS_OK, "70B bf16 config accepted");
    expect(sz.page_bytes == 5242880u, "page of 5,242,880 bytes");
    expect(sz.pool_bytes == static_cast<size_t>(8200) * 5242880u, "pool bytes");
    expect(sz.records_bytes == static_cast<size_t>(8197) * 64u, "64-byte records");
    c.kv_dtype = KVS_KV_FP8_E4M3;
    expect(kvs_required_sizes(&c, &sz) == KVS_OK && sz.page_bytes == 2621440u, "FP8 page of 2,621,440 bytes");
    c.kv_dtype = KVS_KV_KIVI2;
    c.kivi_groups = 4097;
    expect(kvs_required_sizes(&c, &sz) == KVS_OK && sz.group_page_bytes == 80u * 8u * KVS_KIVI_TILE_BYTES,
           "2-bit group page of L*Hkv tiles");
    // every rejected field, one at a time
    struct Bad {
        const char *what;
        void (*edit)(kvs_config &);
    } bad[] = {
        {"block_tokens 8", [](kvs_config &x) { x.block_tokens = 8; }},
        {"head_dim 96", [](kvs_config &x) { x.head_dim = 96; }},
        {"no layers", [](kvs_config &x) { x.num_layers = 0; }},
        {"Hq not a multiple of Hkv", [](kvs_config &x) { x.num_q_heads = 60; }},
        {"16 query heads per KV head", [](kvs_config &x) { x.num_kv_heads = 4; }},
        {"no pool", [](kvs_config &x) { x.pool_blocks = 0; }},
        {"no staging", [](kvs_config &x) { x.staging_pages = 0; }},
        {"layers * pool_blocks past 2^31", [](kvs_config &x) { x.pool_blocks = 1u << 30; }},
        {"alpha above 1", [](kvs_config &x) { x.alpha = 1.5; }},
        {"alpha NaN", [](kvs_config &x) { std::memset(&x.alpha, 0xff, sizeof x.alpha); }},
        {"no recency window", [](kvs_config &x) { x.recency_window = 0; }},
        {"cuts crossed", [](kvs_config &x) { x.cut_lo = 0.7; }},
        {"unknown kv_dtype", [](kvs_config &x) { x.kv_dtype = 9; }},
        {"FP8 at d=64", [](kvs_config &x) { x.kv_dtype = KVS_KV_FP8_E4M3; x.head_dim = 64; }},
        {"FP8 scale 0", [](kvs_config &x) { x.kv_dtype = KVS_KV_FP8_E4M3; x.k_scale = 0.f; }},
        {"2-bit at d=64", [](kvs_config &x) { x.kv_dtype = KVS_KV_KIVI2; x.head_dim = 64; }},
    };
    for (const Bad &b : bad) {
        kvs_config x = base70b();
        b.edit(x);
        const int rc = kvs_required_sizes(&x, &sz);
        expect(rc == KVS_EINVAL, b.what);
        const char *msg = kvs_last_error(nullptr);
        expect(msg && std::strlen(msg) > 0, "a message for the rejected configuration");
    }
    expect(kvs_required_sizes(nullptr, &sz) == KVS_EINVAL, "null config");
}

void plans()
{
    uint64_t seed = 0x6B76;
    for (int call = 0; call < 300; ++call) {
        const uint32_t n = 1 + static_cast<uint32_t>(mix(seed) % 256);
        std::vector<uint32_t> nres(n);
        for (auto &x : nres)
            x = 1 + static_cast<uint32_t>(mix(seed) % 9000);
        const uint32_t L = 1 + static_cast<uint32_t>(mix(seed) % 80);
        const uint32_t H = 1 + static_cast<uint32_t>(mix(seed) % 8);
        const uint32_t workers = 1 + static_cast<uint32_t>(mix(seed) % 1216);
        const uint64_t cap = 1 + mix(seed) % 4000000;
        const uint64_t extra = mix(seed) % 1000;
        uint32_t big = 0, small = 0, tail = 0;
        expect(kvs_debug_chunk_plan(nres.data(), n, L, H, workers, cap, extra, &big, &small, &tail) == KVS_OK,
               "plan call accepted");
        expect(big == 0 || (small > 0 && small <= big), "small chunks no larger than big ones");
    }
    uint32_t a, b, c;
    const uint32_t one = 5;
    expect(kvs_debug_chunk_plan(nullptr, 1, 1, 1, 1, 10, 0, &a, &b, &c) == KVS_EINVAL, "plan: null sizes");
    expect(kvs_debug_chunk_plan(&one, 0, 1, 1, 1, 10, 0, &a, &b, &c) == KVS_EINVAL, "plan: no sequence");
    expect(kvs_debug_chunk_plan(&one, 1, 1, 1, 0, 10, 0, &a, &b, &c) == KVS_EINVAL, "plan: no workers");
}

void create_fails_cleanly()
{
    kvs_ctx_t *ctx = nullptr;
    kvs_config bad = base70b();
    bad.head_dim = 80;
    kvs_buffers buf;
    std::memset(&buf, 0, sizeof buf);
    expect(kvs_create(&bad, &buf, &ctx) == KVS_EINVAL && ctx == nullptr, "create: invalid configuration");
    kvs_config c = base70b();
    expect(kvs_create(&c, nullptr, &ctx) != KVS_OK && ctx == nullptr, "create: no buffers");
    // every buffer named, none usable: creation fails at its first device
    // call (no GPU here) and must release what it took
    static uint8_t fake[4096];
    buf.pool = buf.block_table = buf.records = buf.mass = buf.workspace = buf.staging = fake;
    expect(kvs_create(&c, &buf, &ctx) != KVS_OK && ctx == nullptr, "create: no device");
    expect(kvs_debug_inject(KVS_FAULT_HOSTALLOC, 0) == KVS_OK, "inject a pinned allocation failure");
    expect(kvs_create(&c, &buf, &ctx) != KVS_OK && ctx == nullptr, "create: injected failure");
    expect(kvs_debug_inject(0, 0) == KVS_OK, "clear the injection");
    expect(kvs_debug_inject(1u << 7, 0) == KVS_EINVAL, "unknown injection bit");
    kvs_destroy(nullptr);
    expect(kvs_check_device(nullptr, nullptr) == KVS_EINVAL, "check_device without a context");
    expect(kvs_free_pages(nullptr) == 0 && kvs_step_count(nullptr) == 0, "queries without a context");
}

}  // namespace

int main()
{
    sizes();
    plans();
    create_fails_cleanly();
    if (failures) {
        std::fprintf(stderr, "%d expectation(s) failed\n", failures);
        return 1;
    }
    std::printf("host layer: all expectations hold\n");
    return 0;
}
