// Copy-on-write block copy: duplicate whole physical blocks of the pool.
//
// A block shared by several sequences (reference count > 1) gets a private
// copy before one of them writes into it, and speculative decoding rolls a
// rejected draft back onto such copies (Continuous-Batching-LLM-Inference-
// Engine README, feature list "Paged KV-cache": copy-on-write reference
// counting; "Speculative decoding": KV-cache rollback uses copy-on-write).
//
// One physical block is Hkv * 16 * D contiguous elements in each of K and V
// (plus Hkv scales each for INT8), so a pair is two contiguous runs: each
// thread moves one 16-byte vector of K and of V, grid-stride, fully
// coalesced. Bound: HBM (reads + writes of 2 * Hkv * 16 * D * esize bytes
// per pair).
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

__global__ void copy_blocks_kernel(uint4* __restrict__ k, uint4* __restrict__ v,
                                   float* __restrict__ ks, float* __restrict__ vs,
                                   const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                                   int n_pairs, int vec_per_block, int hkv, int num_blocks,
                                   uint32_t* status) {
    griddep_wait();
    griddep_launch_dependents();
    const long long total = (long long)n_pairs * vec_per_block;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long pair = i / vec_per_block;
        const int c = int(i - pair * vec_per_block);
        const int s = src[pair], d = dst[pair];
        if (unsigned(s) >= unsigned(num_blocks) || unsigned(d) >= unsigned(num_blocks)) {
            if (c == 0) flag_status(status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        if (s == d) continue;
        k[(long long)d * vec_per_block + c] = k[(long long)s * vec_per_block + c];
        v[(long long)d * vec_per_block + c] = v[(long long)s * vec_per_block + c];
        if (ks != nullptr && c < hkv) {
            ks[(long long)d * hkv + c] = ks[(long long)s * hkv + c];
            vs[(long long)d * hkv + c] = vs[(long long)s * hkv + c];
        }
    }
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, float* k_scales,
                                      float* v_scales, const pkv_cache_desc* cache,
                                      const int32_t* src_blocks, const int32_t* dst_blocks,
                                      int32_t num_pairs, uint32_t* dev_status,
                                      cudaStream_t stream) {
    if (!cache || cache->num_blocks <= 0 || cache->num_kv_heads <= 0 || cache->head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache->kv_dtype != PKV_F16 && cache->kv_dtype != PKV_BF16 && cache->kv_dtype != PKV_I8)
        return PKV_ERR_INVALID_ARG;
    if (cache->block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_INVALID_ARG;
    if (!aligned_to(k_cache, 16) || !aligned_to(v_cache, 16) || !aligned_to(src_blocks, 4) ||
        !aligned_to(dst_blocks, 4) || (dev_status && !aligned_to(dev_status, 4)))
        return PKV_ERR_INVALID_ARG;
    const bool i8 = cache->kv_dtype == PKV_I8;
    if (i8 && (!k_scales || !v_scales || !aligned_to(k_scales, 4) || !aligned_to(v_scales, 4)))
        return PKV_ERR_INVALID_ARG;
    const long long block_bytes =
        (long long)cache->num_kv_heads * kBlockSize * cache->head_dim * (i8 ? 1 : 2);
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const long long vpb = block_bytes / 16;
    if (vpb > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    const long long total = (long long)num_pairs * vpb;
    long long grid = (total + kThreads - 1) / kThreads;
    if (grid > 152 * 32) grid = 152 * 32;
    launch_pdl(copy_blocks_kernel, dim3(unsigned(grid)), dim3(kThreads), 0, stream,
               static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
               i8 ? k_scales : nullptr, i8 ? v_scales : nullptr, src_blocks, dst_blocks, num_pairs,
               int(vpb), cache->num_kv_heads, cache->num_blocks, dev_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
