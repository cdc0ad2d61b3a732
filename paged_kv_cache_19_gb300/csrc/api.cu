// api.cu -- host layer of the C ABI: the pool object, argument validation,
// the split-KV plan and kernel launches.  Nothing here allocates or
// synchronises on the append / decode path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <mutex>
#include <new>

#include "kernels.h"
#include "kv_block_manager.h"
#include "kv_mla.h"
#include "kv_paged.h"

struct kv_pool {
    int num_blocks, block_size, kv_heads, head_dim, device;
    kv_dtype dtype;
    size_t elem;            // bytes per cached element
    size_t pool_bytes;      // bytes of the K pool (= bytes of the V pool)
    void* base;             // the single allocation
    uint8_t* k;
    uint8_t* v;
    float* k_scale;
    float* v_scale;
    uint32_t* err;
    CUtensorMap tmk, tmv;   // 5-D tile maps of the K and V pools; latent pools: the map
                            // with the stage box of the producer-warp decode (tmk) and of
                            // the three-CTA decode (tmv)
    CUtensorMap tmt;        // latent pools with blocks of 64: one 128-byte piece of a block
                            // per box (the wide tcgen05 decode)
    CUtensorMap tmh;        // latent pools with blocks of 64: one 128-byte piece of 32 slots
                            // per box (the narrow tcgen05 decode)
    int has_tc;
    int num_sms;
    int mla;                // 1: latent pool (one cached vector per token, no V half)
};

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

constexpr size_t kAlign = 256;
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Failure-path test hook of the decode kernels (kv_debug_decode_stall).
std::atomic<int> g_stop_stage{-1};
std::atomic<unsigned long long> g_consumer_wait_ns{0};

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

bool variant_supported(kv_dtype dtype, int head_dim, int block_size)
{
    if (block_size != 16 && block_size != 32) return false;
    if (dtype == KV_DTYPE_BF16) return head_dim == 64 || head_dim == 128;
    if (dtype == KV_DTYPE_FP8_E4M3) return head_dim == 128;
    return false;
}

// Tile map of one pool half: dims (innermost first) = 128-byte row piece,
// pieces per token row, kv head, slot, block; a box is one block of one kv
// head, written to shared memory with the 128-byte swizzle.
kv_status encode_pool_map(const kv_pool* p, uint8_t* base, CUtensorMap* map, int slots_per_box = 0,
                          int pieces_per_box = 0)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return KV_ERR_CUDA;
    const cuuint64_t row = static_cast<cuuint64_t>(p->head_dim) * p->elem;
    const cuuint64_t per_piece = 128 / p->elem;
    const cuuint64_t dims[5] = {per_piece, row / 128, static_cast<cuuint64_t>(p->kv_heads),
                                static_cast<cuuint64_t>(p->block_size),
                                static_cast<cuuint64_t>(p->num_blocks)};
    const cuuint64_t strides[4] = {128, row, row * p->kv_heads, row * p->kv_heads * p->block_size};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(per_piece),
                               static_cast<cuuint32_t>(pieces_per_box > 0 ? pieces_per_box
                                                                          : row / 128), 1,
                               static_cast<cuuint32_t>(slots_per_box > 0 ? slots_per_box
                                                                         : p->block_size), 1};
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType dt = p->dtype == KV_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = fn(map, dt, 5, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KV_OK : KV_ERR_CUDA;
}

// Tile map of the absorbed queries [batch, q_heads, MLA_DK] (bf16) for the narrow
// tcgen05 decode: dims (innermost first) = number, head, sequence; a box is one 64-number
// piece of min(16, q_heads) heads, written to shared memory with the 128-byte swizzle
// (heads past q_heads read as zeros).
kv_status encode_query_map(const uint16_t* q, int q_heads, int batch, CUtensorMap* map)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return KV_ERR_CUDA;
    const cuuint64_t row = static_cast<cuuint64_t>(kvp::MLA_DK) * 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kvp::MLA_DK), static_cast<cuuint64_t>(q_heads),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {row, row * static_cast<cuuint64_t>(q_heads)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(q_heads < kvp::MLA_TCN_HEADS ? q_heads
                                                                                       : kvp::MLA_TCN_HEADS), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(q), dims, strides, box,
                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KV_OK : KV_ERR_CUDA;
}

struct Plan {
    int group, rows, head_tile, head_groups, split_blocks, max_splits;
    int cta_heads, cta_per_sm;  // kv heads per CTA (1: paged_decode_main), its CTAs per SM
};

// Split-KV plan.  Automatic chunk size: about eight chunks per SM over the
// worst case (every sequence at max_blocks), kept between 64 and 192 blocks --
// long enough that a CTA's start and epilogue are a small part of its life,
// short enough that the last CTAs to start (the remainder chunks, launched
// last) end soon.  Measured on GB300 for the Llama-3-8B-shaped, ragged and
// long-context batches, the best chunks lie between 96 and 256 blocks.
kv_status make_plan(const kv_pool* pl, int batch, int q_heads, int q_len, int max_blocks,
                    int split_tokens, Plan* out)
{
    if (pl == nullptr || batch < 0 || q_heads <= 0 || q_len <= 0 || max_blocks <= 0 ||
        split_tokens < 0)
        return KV_ERR_INVALID_ARG;
    if (q_heads % pl->kv_heads != 0) return KV_ERR_INVALID_ARG;
    if (split_tokens % pl->block_size != 0) return KV_ERR_INVALID_ARG;
    if (static_cast<long long>(max_blocks) * pl->block_size > std::numeric_limits<int>::max())
        return KV_ERR_INVALID_ARG;
    if (static_cast<long long>(q_heads / pl->kv_heads) * q_len > 4096) return KV_ERR_UNSUPPORTED;
    Plan p;
    p.group = q_heads / pl->kv_heads;
    p.rows = p.group * q_len;
    p.head_tile = kvp::head_tile_for_group(p.rows);
    p.head_groups = (p.rows + p.head_tile - 1) / p.head_tile;
    // CTA shape.  With the automatic chunk, decode rows of one tile per kv head run the
    // kernel whose CTA covers a group of kv heads where it is built: two kv heads of a
    // bf16 pool of head_dim 128 and blocks of 16 (three CTAs per SM), four of an fp8 pool
    // of head_dim 128 and blocks of 32 (two per SM) -- measured on GB300 faster than one
    // CTA per kv head with the automatic chunk (Llama-3-8B-shaped layer 95.7 against
    // 99.4-101.1 us; fp8 batch 328 against 334 us).  A chunk given by the caller keeps one
    // CTA per kv head: for the same chunk that grid has more CTAs, which long chunks need
    // to fill the GPU (long-context batch, 4,096-token chunks: 385 against 479 us).
    p.cta_heads = 1;
    p.cta_per_sm = 3;
    if (split_tokens == 0 && p.head_tile == 8) {
        const bool fp8 = pl->dtype == KV_DTYPE_FP8_E4M3;
        const int hc = fp8 ? 4 : 2, ct = fp8 ? 2 : 3;
        if (pl->kv_heads % hc == 0 &&
            kvp::decode_heads_supported(fp8, pl->head_dim, pl->block_size, p.head_tile, hc, ct)) {
            p.cta_heads = hc;
            p.cta_per_sm = ct;
        }
    }
    if (split_tokens > 0) {
        p.split_blocks = split_tokens / pl->block_size;
    } else {
        const long long units = static_cast<long long>(batch > 0 ? batch : 1) * pl->kv_heads *
                                p.head_groups;
        const long long work = units * max_blocks;
        const long long target = static_cast<long long>(pl->num_sms > 0 ? pl->num_sms : 148) * 8;
        long long sb = (work + target - 1) / target;
        // (the two-head CTA measured best at up to 128 blocks on the ragged batch: 201 us
        // at 2,048 tokens against 217 us at 3,072)
        const long long most = p.cta_heads == 2 ? 128 : 192;
        if (sb < 64) sb = 64;
        if (sb > most) sb = most;
        p.split_blocks = static_cast<int>(sb);
    }
    if (p.split_blocks > max_blocks) p.split_blocks = max_blocks;
    p.max_splits = (max_blocks + p.split_blocks - 1) / p.split_blocks;
    if (p.max_splits > 65535) return KV_ERR_UNSUPPORTED;      // grid z limit
    *out = p;
    return KV_OK;
}

// Workspace layout (only when a sequence can have several chunks): partial
// outputs [batch, q_heads, max_splits, d], (max, sum) pairs [batch, q_heads,
// max_splits, 2], then one ticket per (sequence, kv head, head tile).
struct WorkspaceLayout {
    size_t part_o, part_ml, tickets, ticket_bytes, total;
};

WorkspaceLayout workspace_layout(const kv_pool* pl, int batch, const Plan& p)
{
    WorkspaceLayout w{0, 0, 0, 0, 0};
    if (p.max_splits <= 1) return w;
    const size_t n = static_cast<size_t>(batch) * pl->kv_heads * p.rows * p.max_splits;
    w.part_ml = round_up(n * pl->head_dim * sizeof(float), kAlign);
    w.tickets = w.part_ml + round_up(n * 2 * sizeof(float), kAlign);
    w.ticket_bytes = static_cast<size_t>(batch) * pl->kv_heads * p.head_groups * sizeof(int);
    w.total = w.tickets + w.ticket_bytes;
    return w;
}

size_t workspace_bytes_for(const kv_pool* pl, int batch, const Plan& p)
{
    return workspace_layout(pl, batch, p).total;
}

kv_status check_device(const kv_pool* pl)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
    return dev == pl->device ? KV_OK : KV_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int kv_abi_version(void) { return KV_PAGED_ABI_VERSION; }

const char* kv_status_string(kv_status s)
{
    switch (s) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_OUT_OF_MEMORY: return "out of device memory";
    case KV_ERR_OUT_OF_BLOCKS: return "out of KV cache blocks";
    case KV_ERR_UNSUPPORTED: return "unsupported configuration";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

kv_status kv_pool_create(int num_blocks, int block_size, int kv_heads, int head_dim,
                         kv_dtype dtype, int device, kv_pool** out)
{
    if (out == nullptr) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || kv_heads <= 0 || head_dim <= 0 || device < 0)
        return KV_ERR_INVALID_ARG;
    if (dtype != KV_DTYPE_BF16 && dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_INVALID_ARG;
    if (!variant_supported(dtype, head_dim, block_size)) return KV_ERR_UNSUPPORTED;
    const size_t elem = dtype == KV_DTYPE_BF16 ? 2 : 1;
    const long double bytes = static_cast<long double>(num_blocks) * block_size * kv_heads *
                              head_dim * elem;
    if (bytes >= static_cast<long double>(1ull << 40)) return KV_ERR_UNSUPPORTED;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) return KV_ERR_CUDA;
    DeviceGuard guard(device);
    if (!guard.ok) return KV_ERR_CUDA;

    kv_pool* p = new (std::nothrow) kv_pool();
    if (p == nullptr) return KV_ERR_OUT_OF_MEMORY;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->kv_heads = kv_heads;
    p->head_dim = head_dim;
    p->device = device;
    p->dtype = dtype;
    p->elem = elem;
    p->pool_bytes = static_cast<size_t>(bytes);
    const size_t half = round_up(p->pool_bytes, kAlign);
    const size_t scales = round_up(sizeof(float) * kv_heads, kAlign);
    const size_t total = 2 * half + 2 * scales + kAlign;
    if (cudaMalloc(&p->base, total) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return KV_ERR_OUT_OF_MEMORY;
    }
    uint8_t* b = static_cast<uint8_t*>(p->base);
    p->k = b;
    p->v = b + half;
    p->k_scale = reinterpret_cast<float*>(b + 2 * half);
    p->v_scale = reinterpret_cast<float*>(b + 2 * half + scales);
    p->err = reinterpret_cast<uint32_t*>(b + 2 * half + 2 * scales);

    kv_status st = KV_OK;
    if (cudaMemset(p->base, 0, total) != cudaSuccess) st = KV_ERR_CUDA;
    if (st == KV_OK) {
        float* ones = new (std::nothrow) float[kv_heads];
        if (ones == nullptr) {
            st = KV_ERR_OUT_OF_MEMORY;
        } else {
            for (int h = 0; h < kv_heads; ++h) ones[h] = 1.0f;
            if (cudaMemcpy(p->k_scale, ones, sizeof(float) * kv_heads, cudaMemcpyHostToDevice) !=
                    cudaSuccess ||
                cudaMemcpy(p->v_scale, ones, sizeof(float) * kv_heads, cudaMemcpyHostToDevice) !=
                    cudaSuccess)
                st = KV_ERR_CUDA;
            delete[] ones;
        }
    }
    if (st == KV_OK && cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, device) !=
                           cudaSuccess)
        st = KV_ERR_CUDA;
    if (st == KV_OK) st = encode_pool_map(p, p->k, &p->tmk);
    if (st == KV_OK) st = encode_pool_map(p, p->v, &p->tmv);
    if (st == KV_OK) {
        const bool fp8 = dtype == KV_DTYPE_FP8_E4M3;
        for (int nt : {8, 16}) {
            cudaError_t e = fp8 ? kvp::prepare_decode_fp8(head_dim, block_size, nt)
                                : kvp::prepare_decode_bf16(head_dim, block_size, nt);
            if (e != cudaSuccess) st = KV_ERR_CUDA;
        }
        if (kvp::prepare_decode_heads(fp8, head_dim, block_size) != cudaSuccess) st = KV_ERR_CUDA;
    }
    if (st == KV_OK && cudaDeviceSynchronize() != cudaSuccess) st = KV_ERR_CUDA;
    if (st != KV_OK) {
        cudaGetLastError();
        cudaFree(p->base);
        delete p;
        return st;
    }
    *out = p;
    return KV_OK;
}

kv_status kv_pool_destroy(kv_pool* pool)
{
    if (pool == nullptr) return KV_OK;
    kv_status st = KV_OK;
    {
        DeviceGuard guard(pool->device);
        if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) st = KV_ERR_CUDA;
        if (cudaFree(pool->base) != cudaSuccess) st = KV_ERR_CUDA;
    }
    delete pool;
    return st;
}

kv_status kv_pool_tensors(const kv_pool* pool, void** k_pool, void** v_pool, float** k_scale,
                          float** v_scale)
{
    if (pool == nullptr) return KV_ERR_INVALID_ARG;
    if (k_pool) *k_pool = pool->k;
    if (v_pool) *v_pool = pool->v;
    if (k_scale) *k_scale = pool->k_scale;
    if (v_scale) *v_scale = pool->v_scale;
    return KV_OK;
}

kv_status kv_pool_shape(const kv_pool* pool, int* num_blocks, int* block_size, int* kv_heads,
                        int* head_dim, kv_dtype* dtype, int* device)
{
    if (pool == nullptr) return KV_ERR_INVALID_ARG;
    if (num_blocks) *num_blocks = pool->num_blocks;
    if (block_size) *block_size = pool->block_size;
    if (kv_heads) *kv_heads = pool->kv_heads;
    if (head_dim) *head_dim = pool->head_dim;
    if (dtype) *dtype = pool->dtype;
    if (device) *device = pool->device;
    return KV_OK;
}

kv_status kv_pool_set_scales(kv_pool* pool, const float* k_scale_host, const float* v_scale_host)
{
    if (pool == nullptr) return KV_ERR_INVALID_ARG;
    for (const float* s : {k_scale_host, v_scale_host}) {
        if (s == nullptr) continue;
        for (int h = 0; h < pool->kv_heads; ++h)
            if (!(std::isfinite(s[h]) && s[h] > 0.f)) return KV_ERR_INVALID_ARG;
    }
    DeviceGuard guard(pool->device);
    if (!guard.ok) return KV_ERR_CUDA;
    const size_t n = sizeof(float) * pool->kv_heads;
    if (k_scale_host && cudaMemcpy(pool->k_scale, k_scale_host, n, cudaMemcpyHostToDevice) != cudaSuccess)
        return KV_ERR_CUDA;
    if (v_scale_host && cudaMemcpy(pool->v_scale, v_scale_host, n, cudaMemcpyHostToDevice) != cudaSuccess)
        return KV_ERR_CUDA;
    return KV_OK;
}

kv_status kv_pool_device_errors(kv_pool* pool, uint32_t* bits, int clear)
{
    if (pool == nullptr || bits == nullptr) return KV_ERR_INVALID_ARG;
    DeviceGuard guard(pool->device);
    if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) return KV_ERR_CUDA;
    if (cudaMemcpy(bits, pool->err, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KV_ERR_CUDA;
    if (clear && cudaMemset(pool->err, 0, sizeof(uint32_t)) != cudaSuccess) return KV_ERR_CUDA;
    return *bits ? KV_ERR_DEVICE_CHECK : KV_OK;
}

kv_status paged_kv_append(kv_pool* pool, const void* k_new, const void* v_new, int num_tokens,
                          const int32_t* token_seq, const int32_t* token_pos,
                          const int32_t* block_tables, int max_blocks,
                          const int32_t* context_lens, int batch, void* stream)
{
    if (pool == nullptr || num_tokens < 0 || batch < 0 || max_blocks <= 0)
        return KV_ERR_INVALID_ARG;
    if (num_tokens == 0) return KV_OK;
    if (k_new == nullptr || block_tables == nullptr || batch == 0) return KV_ERR_INVALID_ARG;
    if ((v_new == nullptr) != (pool->mla != 0)) return KV_ERR_INVALID_ARG;   // latent pools: no V
    if (token_pos == nullptr && context_lens == nullptr) return KV_ERR_INVALID_ARG;
    if (token_seq == nullptr && num_tokens > batch) return KV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(block_tables, 4) ||
        !aligned(token_seq, 4) || !aligned(token_pos, 4) || !aligned(context_lens, 4))
        return KV_ERR_INVALID_ARG;
    kv_status st = check_device(pool);
    if (st != KV_OK) return st;
    kvp::AppendParams p;
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.token_seq = token_seq;
    p.token_pos = token_pos;
    p.tables = block_tables;
    p.ctx = context_lens;
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.k_scale = pool->k_scale;
    p.v_scale = pool->v_scale;
    p.err = pool->err;
    p.num_tokens = num_tokens;
    p.batch = batch;
    p.max_blocks = max_blocks;
    p.num_blocks = pool->num_blocks;
    p.block_size = pool->block_size;
    p.kv_heads = pool->kv_heads;
    p.head_dim = pool->head_dim;
    p.fp8 = pool->dtype == KV_DTYPE_FP8_E4M3;
    p.q_len = 1;
    return kvp::launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KV_OK
                                                                                   : KV_ERR_CUDA;
}

kv_status kv_copy_blocks(kv_pool* pool, const kv_block_copy* copies, int n, void* stream)
{
    if (pool == nullptr || n < 0) return KV_ERR_INVALID_ARG;
    if (n == 0) return KV_OK;
    if (copies == nullptr || !aligned(copies, 4)) return KV_ERR_INVALID_ARG;
    if (n > (1 << 30)) return KV_ERR_UNSUPPORTED;
    kv_status st = check_device(pool);
    if (st != KV_OK) return st;
    const size_t block_bytes = static_cast<size_t>(pool->block_size) * pool->kv_heads *
                               pool->head_dim * pool->elem;
    return kvp::launch_copy_blocks(copies, n, pool->k, pool->v, block_bytes, pool->num_blocks,
                                   pool->err, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KV_OK
               : KV_ERR_CUDA;
}

kv_status paged_decode_plan(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                            int kv_split_tokens, int* split_tokens, int* max_splits)
{
    Plan p;
    kv_status st = make_plan(pool, batch, q_heads, 1, max_blocks, kv_split_tokens, &p);
    if (st != KV_OK) return st;
    if (split_tokens) *split_tokens = p.split_blocks * pool->block_size;
    if (max_splits) *max_splits = p.max_splits;
    return KV_OK;
}

kv_status kv_debug_decode_stall(int stop_stage, unsigned long long consumer_wait_ns)
{
    if (stop_stage < -1) return KV_ERR_INVALID_ARG;
    g_stop_stage.store(stop_stage, std::memory_order_relaxed);
    g_consumer_wait_ns.store(consumer_wait_ns, std::memory_order_relaxed);
    return KV_OK;
}

kv_status paged_decode_cta_heads(const kv_pool* pool, int batch, int q_heads, int q_len,
                                 int max_blocks, int kv_split_tokens, int* cta_heads)
{
    if (cta_heads == nullptr) return KV_ERR_INVALID_ARG;
    Plan p;
    kv_status st = make_plan(pool, batch, q_heads, q_len, max_blocks, kv_split_tokens, &p);
    if (st != KV_OK) return st;
    *cta_heads = p.cta_heads;
    return KV_OK;
}

kv_status paged_multi_query_workspace_size(const kv_pool* pool, int batch, int q_heads,
                                           int q_len, int max_blocks, int kv_split_tokens,
                                           size_t* bytes)
{
    if (bytes == nullptr) return KV_ERR_INVALID_ARG;
    Plan p;
    kv_status st = make_plan(pool, batch, q_heads, q_len, max_blocks, kv_split_tokens, &p);
    if (st != KV_OK) return st;
    *bytes = workspace_bytes_for(pool, batch, p);
    return KV_OK;
}

kv_status paged_decode_workspace_size(const kv_pool* pool, int batch, int q_heads,
                                      int max_blocks, int kv_split_tokens, size_t* bytes)
{
    return paged_multi_query_workspace_size(pool, batch, q_heads, 1, max_blocks, kv_split_tokens,
                                            bytes);
}

}  // extern "C"

namespace {

// Validates a decode call and fills its kernel parameters and grid (nothing launched).
kv_status make_decode_launch(const kv_pool* pool, const void* q, int q_heads, int q_len,
                             const int32_t* block_tables, int max_blocks,
                             const int32_t* context_lens, int batch, float scale,
                             int kv_split_tokens, void* workspace, size_t workspace_bytes,
                             void* out, float* lse_out, Plan* plan_out, kvp::DecodeParams* pp,
                             dim3* grid)
{
    Plan plan;
    kv_status st = make_plan(pool, batch, q_heads, q_len, max_blocks, kv_split_tokens, &plan);
    if (st != KV_OK) return st;
    if (pool->mla) return KV_ERR_INVALID_ARG;        // latent pools: paged_mla_decode_attention
    if (batch == 0) return KV_OK;
    if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr)
        return KV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4) || !aligned(lse_out, 4) || !aligned(workspace, 16))
        return KV_ERR_INVALID_ARG;
    if (batch > 65535 || static_cast<long long>(pool->kv_heads) * plan.head_groups > 65535)
        return KV_ERR_UNSUPPORTED;                  // grid x / y limits
    const size_t need = workspace_bytes_for(pool, batch, plan);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return KV_ERR_INVALID_ARG;
    st = check_device(pool);
    if (st != KV_OK) return st;

    const WorkspaceLayout wl = workspace_layout(pool, batch, plan);
    kvp::DecodeParams& p = *pp;
    p.q = static_cast<const uint16_t*>(q);
    p.tables = block_tables;
    p.ctx = context_lens;
    p.k_scale = pool->k_scale;
    p.v_scale = pool->v_scale;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse_out;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part_o = need > 0 ? reinterpret_cast<float*>(ws + wl.part_o) : nullptr;
    p.part_ml = need > 0 ? reinterpret_cast<float*>(ws + wl.part_ml) : nullptr;
    p.tickets = need > 0 ? reinterpret_cast<int*>(ws + wl.tickets) : nullptr;
    p.err = pool->err;
    p.batch = batch;
    p.q_heads = q_heads;
    p.kv_heads = pool->kv_heads;
    p.group = plan.group;
    p.head_groups = plan.head_groups;
    p.q_len = q_len;
    p.rows = plan.rows;
    p.max_blocks = max_blocks;
    p.num_blocks = pool->num_blocks;
    p.split_blocks = plan.split_blocks;
    p.max_splits = plan.max_splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_new = nullptr;
    p.v_new = nullptr;
    p.k_pool = nullptr;
    p.v_pool = nullptr;
    p.merge_kernel = 0;
    p.stop_stage = g_stop_stage.load(std::memory_order_relaxed);
    p.consumer_wait_ns = g_consumer_wait_ns.load(std::memory_order_relaxed);
    // chunk-major grid: x = (kv head group, row tile), y = sequence, z = chunk
    *grid = dim3(static_cast<unsigned>(pool->kv_heads / plan.cta_heads * plan.head_groups),
                 static_cast<unsigned>(batch), static_cast<unsigned>(plan.max_splits));
    *plan_out = plan;
    return KV_OK;
}

kv_status launch_decode(const kv_pool* pool, const Plan& plan, dim3 grid, const kvp::DecodeParams& p,
                        void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan.cta_heads > 1) {
        return kvp::launch_decode_heads(pool->dtype == KV_DTYPE_FP8_E4M3, pool->head_dim,
                                        pool->block_size, plan.head_tile, plan.cta_heads,
                                        plan.cta_per_sm, grid, pool->tmk, pool->tmv, p, s) == cudaSuccess
                   ? KV_OK
                   : KV_ERR_CUDA;
    }
    cudaError_t e = pool->dtype == KV_DTYPE_BF16
                        ? kvp::launch_decode_bf16(pool->head_dim, pool->block_size, plan.head_tile,
                                                  grid, pool->tmk, pool->tmv, p, s)
                        : kvp::launch_decode_fp8(pool->head_dim, pool->block_size, plan.head_tile,
                                                 grid, pool->tmk, pool->tmv, p, s);
    return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // namespace

extern "C" {

kv_status paged_attention_multi_query(const kv_pool* pool, const void* q, int q_heads, int q_len,
                                      const int32_t* block_tables, int max_blocks,
                                      const int32_t* context_lens, int batch, float scale,
                                      int kv_split_tokens, void* workspace,
                                      size_t workspace_bytes, void* out, float* lse_out,
                                      void* stream)
{
    Plan plan;
    kvp::DecodeParams p;
    dim3 grid;
    const kv_status st = make_decode_launch(pool, q, q_heads, q_len, block_tables, max_blocks,
                                            context_lens, batch, scale, kv_split_tokens, workspace,
                                            workspace_bytes, out, lse_out, &plan, &p, &grid);
    if (st != KV_OK || batch == 0) return st;
    return launch_decode(pool, plan, grid, p, stream);
}

kv_status paged_decode_step(kv_pool* pool, const void* k_new, const void* v_new, const void* q,
                            int q_heads, int q_len, const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, int batch, float scale,
                            int kv_split_tokens, void* workspace, size_t workspace_bytes,
                            void* out, float* lse_out, void* stream)
{
    if (pool == nullptr || q_len < 1) return KV_ERR_INVALID_ARG;
    // everything is checked before anything is launched
    Plan plan;
    kvp::DecodeParams p;
    dim3 grid;
    kv_status st = make_decode_launch(pool, q, q_heads, q_len, block_tables, max_blocks,
                                      context_lens, batch, scale, kv_split_tokens, workspace,
                                      workspace_bytes, out, lse_out, &plan, &p, &grid);
    if (st != KV_OK || batch == 0) return st;
    if (k_new == nullptr || v_new == nullptr || !aligned(k_new, 16) || !aligned(v_new, 16))
        return KV_ERR_INVALID_ARG;
    if (static_cast<long long>(batch) * q_len > std::numeric_limits<int>::max())
        return KV_ERR_UNSUPPORTED;
    if (plan.head_tile == 8) {
        // One kernel: the CTA that reads a block holding one of the step's new tokens writes
        // that token's rows of its kv heads into the pool first (the append's arithmetic, the
        // same bytes), so no append kernel has to finish before the attention starts.
        p.k_new = static_cast<const uint16_t*>(k_new);
        p.v_new = static_cast<const uint16_t*>(v_new);
        p.k_pool = pool->k;
        p.v_pool = pool->v;
        return launch_decode(pool, plan, grid, p, stream);
    }
    // 16-row tiles: the append kernel, then the attention (the kernel's step form is not
    // built for them)
    kvp::AppendParams a;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.token_seq = nullptr;
    a.token_pos = nullptr;
    a.tables = block_tables;
    a.ctx = context_lens;
    a.k_pool = pool->k;
    a.v_pool = pool->v;
    a.k_scale = pool->k_scale;
    a.v_scale = pool->v_scale;
    a.err = pool->err;
    a.num_tokens = batch * q_len;
    a.batch = batch;
    a.max_blocks = max_blocks;
    a.num_blocks = pool->num_blocks;
    a.block_size = pool->block_size;
    a.kv_heads = pool->kv_heads;
    a.head_dim = pool->head_dim;
    a.fp8 = pool->dtype == KV_DTYPE_FP8_E4M3;
    a.q_len = q_len;
    if (kvp::launch_append(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KV_ERR_CUDA;
    return launch_decode(pool, plan, grid, p, stream);
}

kv_status paged_decode_attention(const kv_pool* pool, const void* q, int q_heads,
                                 const int32_t* block_tables, int max_blocks,
                                 const int32_t* context_lens, int batch, float scale,
                                 int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                 void* out, float* lse_out, void* stream)
{
    return paged_attention_multi_query(pool, q, q_heads, 1, block_tables, max_blocks,
                                       context_lens, batch, scale, kv_split_tokens, workspace,
                                       workspace_bytes, out, lse_out, stream);
}

kv_status paged_merge_attention_states(const void* outs, const float* lses, int n_src, long long rows,
                                       int head_dim, void* out, float* lse_out, void* stream)
{
    if (n_src < 1 || rows < 0 || head_dim < 8 || head_dim > 1024 || head_dim % 8 != 0)
        return KV_ERR_INVALID_ARG;
    if (rows == 0) return KV_OK;
    if (outs == nullptr || lses == nullptr || out == nullptr) return KV_ERR_INVALID_ARG;
    if (!aligned(outs, 16) || !aligned(out, 16) || !aligned(lses, 4) || !aligned(lse_out, 4))
        return KV_ERR_INVALID_ARG;
    return kvp::launch_merge_attention_states(
               static_cast<const uint16_t*>(outs), lses, n_src, rows, head_dim,
               static_cast<uint16_t*>(out), lse_out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KV_OK
               : KV_ERR_CUDA;
}

kv_status paged_decode_attention_split_merge(const kv_pool* pool, const void* q, int q_heads,
                                             const int32_t* block_tables, int max_blocks,
                                             const int32_t* context_lens, int batch, float scale,
                                             int kv_split_tokens, void* workspace,
                                             size_t workspace_bytes, void* out, float* lse_out,
                                             void* stream)
{
    Plan plan;
    kvp::DecodeParams p;
    dim3 grid;
    const kv_status st = make_decode_launch(pool, q, q_heads, 1, block_tables, max_blocks,
                                            context_lens, batch, scale, kv_split_tokens, workspace,
                                            workspace_bytes, out, lse_out, &plan, &p, &grid);
    if (st != KV_OK || batch == 0) return st;
    p.merge_kernel = plan.max_splits > 1;
    kv_status r = launch_decode(pool, plan, grid, p, stream);
    if (r != KV_OK || !p.merge_kernel) return r;
    return kvp::launch_decode_merge(p, pool->head_dim, pool->block_size,
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KV_OK
               : KV_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Multi-head latent attention (absorbed form) over a latent pool.
// ---------------------------------------------------------------------------
namespace {

constexpr int kMlaHeadTile = 16;

// The three forms of the latent decode.
enum MlaForm {
    kMlaMma = 0,            // mma.sync, head tiles of 16, a CTA per (tile, sequence, chunk)
    kMlaWide = 1,           // tcgen05, head tiles of 128, two latent halves each
    kMlaNarrow = 2,         // tcgen05, head tiles of 16
};

struct MlaPlan {
    int head_tiles, split_blocks, max_splits;
    int form;               // MlaForm
};

// Blocks of 64 tokens take a tcgen05 form: the wide one for at least 64 heads (tiles of
// 128 rows), the narrow one below that.
int mla_form(const kv_pool* pl, int q_heads)
{
    if (!pl->has_tc) return kMlaMma;
    return q_heads >= 64 ? kMlaWide : kMlaNarrow;
}

// Automatic chunk: about eight chunks per SM over the worst case, kept between
// 768 and 2048 tokens.  Measured on GB300 (DeepSeek-shaped layer, contexts
// uniform in [512, 4096]): 16 heads are fastest with 768-token chunks (about
// 2.5 CTAs per SM), 128 heads with ~1700 (chunks of 512 pay too many merges).
kv_status make_mla_plan(const kv_pool* pl, int batch, int q_heads, int max_blocks,
                        int split_tokens, MlaPlan* out)
{
    if (pl == nullptr || !pl->mla || batch < 0 || q_heads <= 0 || max_blocks <= 0 ||
        split_tokens < 0)
        return KV_ERR_INVALID_ARG;
    if (split_tokens % pl->block_size != 0) return KV_ERR_INVALID_ARG;
    if (static_cast<long long>(max_blocks) * pl->block_size > std::numeric_limits<int>::max())
        return KV_ERR_INVALID_ARG;
    MlaPlan p;
    p.form = mla_form(pl, q_heads);
    const int tile = p.form == kMlaWide ? kvp::MLA_TC_HEADS : kMlaHeadTile;
    p.head_tiles = (q_heads + tile - 1) / tile;
    if (p.form != kMlaMma) {
        // the units ((latent half,) head tile, sequence, block) are cut into one contiguous
        // range per CTA; split_blocks is the least a range holds (the chunk argument, or
        // automatically about half the worst-case share of an SM, 4..16 blocks), so a
        // sequence of max_blocks blocks is cut into at most ceil((max_blocks - 1) /
        // split_blocks) + 1 pieces, each merged from its own partial
        const int outer = p.head_tiles * (p.form == kMlaWide ? 2 : 1);
        if (split_tokens > 0) {
            p.split_blocks = split_tokens / pl->block_size;
        } else {
            const long long units = static_cast<long long>(batch > 0 ? batch : 1) * outer * max_blocks;
            const long long share = units / (2LL * (pl->num_sms > 0 ? pl->num_sms : 148));
            p.split_blocks = static_cast<int>(share < 4 ? 4 : (share > 16 ? 16 : share));
        }
        if (p.split_blocks > max_blocks) p.split_blocks = max_blocks;
        p.max_splits = (max_blocks - 1 + p.split_blocks - 1) / p.split_blocks + 1;
        if (p.max_splits > max_blocks) p.max_splits = max_blocks;
        // the partition's arithmetic: units x CTAs must stay far inside 64 bits
        const long long units_max = static_cast<long long>(batch) * outer * max_blocks;
        if (units_max > (1LL << 40)) return KV_ERR_UNSUPPORTED;
        if (p.max_splits > 65535 || p.head_tiles > 32767 || batch > 65535) return KV_ERR_UNSUPPORTED;
        *out = p;
        return KV_OK;
    }
    if (split_tokens > 0) {
        p.split_blocks = split_tokens / pl->block_size;
    } else {
        const long long units = static_cast<long long>(batch > 0 ? batch : 1) * p.head_tiles;
        const long long work = units * max_blocks * pl->block_size;
        const long long target = static_cast<long long>(pl->num_sms > 0 ? pl->num_sms : 148) * 8;
        long long tok = (work + target - 1) / target;
        if (tok < 768) tok = 768;
        if (tok > 2048) tok = 2048;
        p.split_blocks = static_cast<int>((tok + pl->block_size - 1) / pl->block_size);
    }
    if (p.split_blocks > max_blocks) p.split_blocks = max_blocks;
    p.max_splits = (max_blocks + p.split_blocks - 1) / p.split_blocks;
    if (p.max_splits > 65535 || p.head_tiles > 65535 || batch > 65535) return KV_ERR_UNSUPPORTED;
    *out = p;
    return KV_OK;
}

// partial outputs [batch, q_heads, max_splits, 512], (max, sum) pairs, then one ticket
// per (sequence, head tile); the tensor-core form lays its pieces out per (sequence,
// head tile, latent half, split) instead.
WorkspaceLayout mla_workspace_layout(int batch, int q_heads, const MlaPlan& p)
{
    WorkspaceLayout w{0, 0, 0, 0, 0};
    if (p.max_splits > 1 && p.form == kMlaNarrow) {
        // pieces (sequence, head tile, split): fp16 partials of 16 heads x 512 latent
        // numbers, fp32 (max, sum) per head, then the piece count of each (sequence, head tile)
        const size_t pieces = static_cast<size_t>(batch) * p.head_tiles * p.max_splits;
        w.part_ml = round_up(pieces * kvp::MLA_TCN_HEADS * kvp::MLA_DV * 2, kAlign);
        w.tickets = w.part_ml + round_up(pieces * kvp::MLA_TCN_HEADS * 2 * sizeof(float), kAlign);
        w.ticket_bytes = static_cast<size_t>(batch) * p.head_tiles * sizeof(int);
        w.total = w.tickets + w.ticket_bytes;
    } else if (p.max_splits > 1 && p.form == kMlaWide) {
        // pieces (sequence, head tile, latent half, split): fp16 partials of 128 heads x
        // 256 latent numbers, fp32 (max, sum) per head, then the piece count of each
        // (sequence, head tile, half) -- read by the merge kernel
        const size_t pieces = static_cast<size_t>(batch) * p.head_tiles * 2 * p.max_splits;
        w.part_ml = round_up(pieces * kvp::MLA_TC_HEADS * (kvp::MLA_DV / 2) * 2, kAlign);
        w.tickets = w.part_ml + round_up(pieces * kvp::MLA_TC_HEADS * 2 * sizeof(float), kAlign);
        w.ticket_bytes = static_cast<size_t>(batch) * p.head_tiles * 2 * sizeof(int);
        w.total = w.tickets + w.ticket_bytes;
    } else if (p.max_splits > 1) {
        const size_t n = static_cast<size_t>(batch) * q_heads * p.max_splits;
        w.part_ml = round_up(n * kvp::MLA_DV * sizeof(float), kAlign);
        w.tickets = w.part_ml + round_up(n * 2 * sizeof(float), kAlign);
        w.ticket_bytes = static_cast<size_t>(batch) * p.head_tiles * sizeof(int);
        w.total = w.tickets + w.ticket_bytes;
    }
    return w;
}

}  // namespace

extern "C" {

kv_status kv_mla_pool_create(int num_blocks, int block_size, int latent_dim, int rope_dim,
                             int device, kv_pool** out)
{
    if (out == nullptr) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || latent_dim <= 0 || rope_dim < 0 || device < 0)
        return KV_ERR_INVALID_ARG;
    if (latent_dim != kvp::MLA_DV || rope_dim != kvp::MLA_DR) return KV_ERR_UNSUPPORTED;
    if (kvp::mla_stage_tokens(block_size, true) == 0) return KV_ERR_UNSUPPORTED;
    const long double bytes = static_cast<long double>(num_blocks) * block_size * kvp::MLA_DK * 2;
    if (bytes >= static_cast<long double>(1ull << 40)) return KV_ERR_UNSUPPORTED;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) return KV_ERR_CUDA;
    DeviceGuard guard(device);
    if (!guard.ok) return KV_ERR_CUDA;

    kv_pool* p = new (std::nothrow) kv_pool();
    if (p == nullptr) return KV_ERR_OUT_OF_MEMORY;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->kv_heads = 1;
    p->head_dim = kvp::MLA_DK;
    p->device = device;
    p->dtype = KV_DTYPE_BF16;
    p->elem = 2;
    p->mla = 1;
    p->pool_bytes = static_cast<size_t>(bytes);
    const size_t half = round_up(p->pool_bytes, kAlign);
    const size_t scales = round_up(sizeof(float), kAlign);
    const size_t total = half + 2 * scales + kAlign;
    if (cudaMalloc(&p->base, total) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return KV_ERR_OUT_OF_MEMORY;
    }
    uint8_t* b = static_cast<uint8_t*>(p->base);
    p->k = b;
    p->v = nullptr;
    p->k_scale = reinterpret_cast<float*>(b + half);
    p->v_scale = reinterpret_cast<float*>(b + half + scales);
    p->err = reinterpret_cast<uint32_t*>(b + half + 2 * scales);
    kv_status st = KV_OK;
    if (cudaMemset(p->base, 0, total) != cudaSuccess) st = KV_ERR_CUDA;
    if (st == KV_OK && cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, device) !=
                           cudaSuccess)
        st = KV_ERR_CUDA;
    if (st == KV_OK)
        st = encode_pool_map(p, p->k, &p->tmk, kvp::mla_stage_tokens(block_size, true));
    if (st == KV_OK)
        st = encode_pool_map(p, p->k, &p->tmv, kvp::mla_stage_tokens(block_size, false));
    if (st == KV_OK && block_size == kvp::MLA_TC_BLOCK) {
        st = encode_pool_map(p, p->k, &p->tmt, block_size, 1);
        if (st == KV_OK) st = encode_pool_map(p, p->k, &p->tmh, kvp::MLA_TCN_STAGE_TOKENS, 1);
        if (st == KV_OK && kvp::prepare_mla_decode_tc() != cudaSuccess) st = KV_ERR_CUDA;
        if (st == KV_OK && kvp::prepare_mla_decode_tcn() != cudaSuccess) st = KV_ERR_CUDA;
        p->has_tc = 1;
    }
    if (st == KV_OK && kvp::prepare_mla_decode(block_size) != cudaSuccess) st = KV_ERR_CUDA;
    if (st == KV_OK && cudaDeviceSynchronize() != cudaSuccess) st = KV_ERR_CUDA;
    if (st != KV_OK) {
        cudaGetLastError();
        cudaFree(p->base);
        delete p;
        return st;
    }
    *out = p;
    return KV_OK;
}

kv_status paged_mla_decode_plan(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                                int kv_split_tokens, int* split_tokens, int* max_splits)
{
    MlaPlan p;
    kv_status st = make_mla_plan(pool, batch, q_heads, max_blocks, kv_split_tokens, &p);
    if (st != KV_OK) return st;
    if (split_tokens) *split_tokens = p.split_blocks * pool->block_size;
    if (max_splits) *max_splits = p.max_splits;
    return KV_OK;
}

kv_status paged_mla_workspace_size(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                                   int kv_split_tokens, size_t* bytes)
{
    if (bytes == nullptr) return KV_ERR_INVALID_ARG;
    MlaPlan p;
    kv_status st = make_mla_plan(pool, batch, q_heads, max_blocks, kv_split_tokens, &p);
    if (st != KV_OK) return st;
    *bytes = mla_workspace_layout(batch, q_heads, p).total;
    return KV_OK;
}

}  // extern "C"

namespace {

// Everything paged_mla_decode_attention checks and sets up before its launch.
kv_status make_mla_launch(const kv_pool* pool, const void* q, int q_heads, const int32_t* block_tables,
                          int max_blocks, const int32_t* context_lens, int batch, float scale,
                          int kv_split_tokens, void* workspace, size_t workspace_bytes, void* out,
                          float* lse_out, MlaPlan* plan_out, kvp::MlaParams* params)
{
    MlaPlan plan;
    kv_status st = make_mla_plan(pool, batch, q_heads, max_blocks, kv_split_tokens, &plan);
    if (st != KV_OK) return st;
    if (batch == 0) return KV_OK;
    if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr)
        return KV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4) || !aligned(lse_out, 4) || !aligned(workspace, 16))
        return KV_ERR_INVALID_ARG;
    const WorkspaceLayout wl = mla_workspace_layout(batch, q_heads, plan);
    if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total))
        return KV_ERR_INVALID_ARG;
    st = check_device(pool);
    if (st != KV_OK) return st;

    kvp::MlaParams& p = *params;
    p.q = static_cast<const uint16_t*>(q);
    p.tables = block_tables;
    p.ctx = context_lens;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse_out;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part_o = wl.total > 0 ? reinterpret_cast<float*>(ws + wl.part_o) : nullptr;
    p.part_ml = wl.total > 0 ? reinterpret_cast<float*>(ws + wl.part_ml) : nullptr;
    p.tickets = wl.total > 0 ? reinterpret_cast<int*>(ws + wl.tickets) : nullptr;
    p.err = pool->err;
    p.batch = batch;
    p.q_heads = q_heads;
    p.head_tiles = plan.head_tiles;
    p.max_blocks = max_blocks;
    p.num_blocks = pool->num_blocks;
    p.split_blocks = plan.split_blocks;
    p.max_splits = plan.max_splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_new = nullptr;
    p.pool = nullptr;
    *plan_out = plan;
    return KV_OK;
}

kv_status launch_mla(const kv_pool* pool, const MlaPlan& plan, const kvp::MlaParams& p, void* stream)
{
    if (plan.form != kMlaMma) {
        // persistent: one CTA per SM, each taking a contiguous range of the units
        // ((latent half,) head tile, sequence, block); no more CTAs than ranges of
        // split_blocks units the longest batch could have
        const int outer = plan.head_tiles * (plan.form == kMlaWide ? 2 : 1);
        const long long units_max = static_cast<long long>(outer) * p.batch * p.max_blocks;
        const long long ranges = units_max / plan.split_blocks > 0 ? units_max / plan.split_blocks : 1;
        const int sms = pool->num_sms > 0 ? pool->num_sms : 148;
        const dim3 grid(static_cast<unsigned>(ranges < sms ? ranges : sms));
        if (plan.form == kMlaWide)
            return kvp::launch_mla_decode_tc(grid, pool->tmt, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
                       ? KV_OK
                       : KV_ERR_CUDA;
        CUtensorMap tq;
        const kv_status st = encode_query_map(p.q, p.q_heads, p.batch, &tq);
        if (st != KV_OK) return st;
        return kvp::launch_mla_decode_tcn(grid, pool->tmh, tq, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? KV_OK
                   : KV_ERR_CUDA;
    }
    // chunk-major grid: x = head tile, y = sequence, z = chunk.  Grids of up to
    // three CTAs per SM run the producer-warp variant (32-token stages, two CTAs
    // per SM), larger ones the three-CTAs-per-SM variant (16-token stages).
    const dim3 grid(static_cast<unsigned>(plan.head_tiles), static_cast<unsigned>(p.batch),
                    static_cast<unsigned>(plan.max_splits));
    const long long ctas = static_cast<long long>(plan.head_tiles) * p.batch * plan.max_splits;
    const bool prod = ctas <= 3LL * (pool->num_sms > 0 ? pool->num_sms : 148);
    return kvp::launch_mla_decode(pool->block_size, prod, grid, prod ? pool->tmk : pool->tmv, p,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KV_OK
               : KV_ERR_CUDA;
}

}  // namespace

extern "C" {

kv_status paged_mla_decode_attention(const kv_pool* pool, const void* q, int q_heads,
                                     const int32_t* block_tables, int max_blocks,
                                     const int32_t* context_lens, int batch, float scale,
                                     int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                     void* out, float* lse_out, void* stream)
{
    MlaPlan plan;
    kvp::MlaParams p;
    kv_status st = make_mla_launch(pool, q, q_heads, block_tables, max_blocks, context_lens, batch, scale,
                                   kv_split_tokens, workspace, workspace_bytes, out, lse_out, &plan, &p);
    if (st != KV_OK || batch == 0) return st;
    return launch_mla(pool, plan, p, stream);
}

kv_status paged_mla_decode_step(kv_pool* pool, const void* kv_new, const void* q, int q_heads,
                                const int32_t* block_tables, int max_blocks,
                                const int32_t* context_lens, int batch, float scale,
                                int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                void* out, float* lse_out, void* stream)
{
    if (pool == nullptr) return KV_ERR_INVALID_ARG;
    // everything is checked before anything is launched
    MlaPlan plan;
    kvp::MlaParams p;
    kv_status st = make_mla_launch(pool, q, q_heads, block_tables, max_blocks, context_lens, batch, scale,
                                   kv_split_tokens, workspace, workspace_bytes, out, lse_out, &plan, &p);
    if (st != KV_OK || batch == 0) return st;
    if (kv_new == nullptr || !aligned(kv_new, 16)) return KV_ERR_INVALID_ARG;
    // One attention launch (plus the merge of cut sequences): the CTA that reads the block
    // holding a sequence's new vector writes it into the pool first (the append's bytes).
    p.kv_new = static_cast<const uint16_t*>(kv_new);
    p.pool = pool->k;
    return launch_mla(pool, plan, p, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode attention.
//
// For callers that cannot allocate device memory themselves: plug-in hosts
// that hand a kernel only its input and output buffers, engines whose own
// allocator has reserved the whole GPU up front, and latency-critical paths
// where cudaMalloc's implicit device-wide synchronisation would stall other
// streams.  The split-KV partials live in the fixed-size array below, which is
// part of the library's device image: every GPU that loads the library holds
// it until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char kv_noalloc_scratch[KV_NO_ALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// Looked up once per device; the lookup is the only set-up step.
kv_status scratch_address(int device, void** addr)
{
    if (device < 0 || device >= kMaxScratchDevices) return KV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[device] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, kv_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return KV_ERR_CUDA;
        }
        g_scratch_addr[device] = p;
    }
    *addr = g_scratch_addr[device];
    return KV_OK;
}

}  // namespace

extern "C" kv_status paged_decode_attention_noalloc(const kv_pool* pool, const void* q, int q_heads,
                                                    const int32_t* block_tables, int max_blocks,
                                                    const int32_t* context_lens, int batch,
                                                    float scale, int kv_split_tokens, void* out,
                                                    float* lse_out, void* stream)
{
    Plan plan;
    kv_status st = make_plan(pool, batch, q_heads, 1, max_blocks, kv_split_tokens, &plan);
    if (st != KV_OK) return st;
    if (batch == 0) return KV_OK;
    const size_t need = workspace_bytes_for(pool, batch, plan);
    if (need > KV_NO_ALLOC_SCRATCH_BYTES) return KV_ERR_UNSUPPORTED;
    st = check_device(pool);
    if (st != KV_OK) return st;
    void* scratch = nullptr;
    if (need > 0) {
        st = scratch_address(pool->device, &scratch);
        if (st != KV_OK) return st;
    }
    // Every argument is checked before the shared array is touched: a call that is
    // rejected writes nothing to it and launches nothing.
    kvp::DecodeParams p;
    dim3 grid;
    st = make_decode_launch(pool, q, q_heads, 1, block_tables, max_blocks, context_lens, batch,
                            scale, kv_split_tokens, scratch, need, out, lse_out, &plan, &p, &grid);
    if (st != KV_OK) return st;
    if (need > 0) {
        // The per-unit chunk counts in the scratch must start at zero, whatever
        // an earlier (possibly failed) call left there.
        const WorkspaceLayout wl = workspace_layout(pool, batch, plan);
        if (wl.ticket_bytes > 0 &&
            cudaMemsetAsync(static_cast<uint8_t*>(scratch) + wl.tickets, 0, wl.ticket_bytes,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            cudaGetLastError();
            return KV_ERR_CUDA;
        }
    }
    return launch_decode(pool, plan, grid, p, stream);
}
