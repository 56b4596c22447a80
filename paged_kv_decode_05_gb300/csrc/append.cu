// KV append (cache write): scatter new K/V rows into the paged block pool.
//
// The forward pass writes each step's K/V into the paged cache through a slot
// mapping (mini-inference-engine, Connections "Llama forward -> Paged KV
// cache: writes and reads"; low-latency-distributed-llm-serving-infrastructure,
// Connections "LLM engine -> KV cache manager: writes KV cache", "Paged
// attention -> KV cache manager: maps cache slots"), optionally as INT8
// (paged-inference-engine overview, "paged INT8 KV storage").
//
// fp16/bf16: one 16-byte vector per thread, a bit copy.
// INT8: two stream-ordered kernels over (token, kv_head) warps, so that every
// (block, kv_head) tile sees all of a call's new rows before its scale is set:
//   gather -> per tile: atomicMax of each new row's |x| max (K and V), an
//             owner claim (the call's first token in the tile), the set of
//             rows the call writes and each such row's token index
//   settle -> the owning warp alone sets the tile's scale, requantises the
//             stored codes when the scale grows, encodes every new row of
//             the tile under the final scale and clears the tile's scratch,
//             so the workspace is zero again for the next call
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void append_copy_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                   const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                                   uint4* __restrict__ v_cache, int n_tokens, int hkv,
                                   int vec_per_row, long long pool_slots, uint32_t* status) {
    griddep_wait();
    griddep_launch_dependents();
    const long long per_tok = (long long)hkv * vec_per_row;
    const long long total = (long long)n_tokens * per_tok;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long n = i / per_tok;
        const long long rem = i - n * per_tok;           // kvh * vec_per_row + c
        const long long slot = slots[n];
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (rem == 0) flag_status(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const long long kvh = rem / vec_per_row;
        const long long c = rem - kvh * vec_per_row;
        const long long blk = slot / kBlockSize, row = slot % kBlockSize;
        const long long dst = ((blk * hkv + kvh) * kBlockSize + row) * vec_per_row + c;
        k_cache[dst] = k_new[i];
        v_cache[dst] = v_new[i];
    }
}

// ---------------------------------------------------------------- INT8 ---
// Per-tile scratch: absmax bits of K and of V, the owner claim N - n of the
// call's first token in the tile, and the mask of rows the call writes; all
// zero between calls. Beside it, the token index of each row the call writes.
struct TileScratch {
    uint32_t amax_k, amax_v, owner, rows;
};

struct I8Args {
    const void* k_new;
    const void* v_new;
    const int64_t* slots;
    int8_t* k_cache;
    int8_t* v_cache;
    float* k_scales;
    float* v_scales;
    TileScratch* tiles;   // [num_blocks * hkv]
    int32_t* row_tok;     // [num_blocks * hkv * 16]
    uint32_t* status;
    int n_tokens;
    int hkv;
    long long pool_slots;
};

// Item = (token n, kv head), one warp each. Returns the tile index or -1.
__device__ __forceinline__ long long item_tile(const I8Args& a, long long item, long long* n_out,
                                               int* row_out, bool flag) {
    const long long n = item / a.hkv;
    const int kvh = int(item - n * a.hkv);
    const long long slot = a.slots[n];
    *n_out = n;
    if (slot < 0) return -1;
    if (slot >= a.pool_slots) {
        if (flag && kvh == 0 && (threadIdx.x & 31) == 0) flag_status(a.status, PKV_DEV_BAD_SLOT);
        return -1;
    }
    *row_out = int(slot % kBlockSize);
    return (slot / kBlockSize) * a.hkv + kvh;
}

template <typename S, int D>
__device__ __forceinline__ void load_row(const void* src, long long row_elem0, float* x) {
    constexpr int EPL = D / 32;  // elements per lane
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[e] = load_scalar(S{}, src, row_elem0 + lane * EPL + e);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

template <typename S, int D>
__global__ void i8_gather_kernel(I8Args a) {
    griddep_wait();
    griddep_launch_dependents();
    const long long items = (long long)a.n_tokens * a.hkv;
    for (long long it = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; it < items;
         it += ((long long)gridDim.x * blockDim.x) >> 5) {
        // the new rows are loaded while the slot is resolved
        float xk[D / 32], xv[D / 32];
        load_row<S, D>(a.k_new, it * D, xk);
        load_row<S, D>(a.v_new, it * D, xv);
        long long n;
        int row;
        const long long t = item_tile(a, it, &n, &row, true);
        if (t < 0) continue;
        float mk = 0.f, mv = 0.f;
#pragma unroll
        for (int e = 0; e < D / 32; ++e) {
            mk = fmaxf(mk, fabsf(xk[e]));
            mv = fmaxf(mv, fabsf(xv[e]));
        }
        mk = warp_max(mk);
        mv = warp_max(mv);
        if ((threadIdx.x & 31) == 0) {
            TileScratch* ts = a.tiles + t;
            // non-negative floats order like their bit patterns
            atomicMax(&ts->amax_k, __float_as_uint(mk));
            atomicMax(&ts->amax_v, __float_as_uint(mv));
            atomicMax(&ts->owner, uint32_t(a.n_tokens - n));
            atomicOr(&ts->rows, 1u << row);
            a.row_tok[t * kBlockSize + row] = int32_t(n);
        }
    }
}

// The tile's scale from the call's absmax and the stored scale s_o (0 = never
// written): s_c = a / 127 (IEEE division); s = s_c if s_o == 0, s_o if
// s_c <= s_o, else s_c (the tile's stored codes are then requantised).
__device__ __forceinline__ float settle_scale(uint32_t amax_bits, float s_o, bool* grow) {
    const float s_c = __fdiv_rn(__uint_as_float(amax_bits), 127.0f);
    *grow = (s_o != 0.f) && !(s_c <= s_o);
    return (s_o != 0.f && s_c <= s_o) ? s_o : s_c;
}

__device__ __forceinline__ uint4 requant_vec(const uint4& in, float s_o, float s) {
    return make_uint4(requant_word(in.x, s_o, s), requant_word(in.y, s_o, s),
                      requant_word(in.z, s_o, s), requant_word(in.w, s_o, s));
}

template <int EPL>
__device__ __forceinline__ void store_codes(int8_t* cache, long long dst, const float* x, float s) {
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) packed |= (uint32_t(quant_code(x[e], s)) & 0xffu) << (8 * e);
    if (EPL == 4) *reinterpret_cast<uint32_t*>(cache + dst) = packed;
    else *reinterpret_cast<uint16_t*>(cache + dst) = uint16_t(packed);
}

// Re-express every stored code of one tile under a grown scale: each lane
// loads all its 16-byte words before storing any, so the tile costs one
// memory round trip.
template <int D>
__device__ __forceinline__ void requant_tile(int8_t* tile, float s_o, float s, int lane) {
    constexpr int V4 = kBlockSize * D / 16 / 32;   // 16-byte words of a tile per lane
    uint4* w = reinterpret_cast<uint4*>(tile);
    uint4 c[V4];
#pragma unroll
    for (int i = 0; i < V4; ++i) c[i] = w[lane + 32 * i];
#pragma unroll
    for (int i = 0; i < V4; ++i) w[lane + 32 * i] = requant_vec(c[i], s_o, s);
}

// One warp per tile (the warp of the call's first token in it) settles the
// K and V scales, requantises a tile whose scale grew, and encodes the call's
// new rows under the final scales. The first new row and the stored scales
// are loaded together, before the scales are settled, to shorten the chain
// of dependent memory accesses.
template <typename S, int D>
__global__ void __launch_bounds__(kThreads, 4) i8_settle_kernel(I8Args a) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int EPL = D / 32;
    const long long items = (long long)a.n_tokens * a.hkv;
    const int lane = threadIdx.x & 31;
    for (long long it = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; it < items;
         it += ((long long)gridDim.x * blockDim.x) >> 5) {
        long long n;
        int row;
        const long long t = item_tile(a, it, &n, &row, false);
        if (t < 0) continue;
        TileScratch* ts = a.tiles + t;
        const TileScratch sc = *ts;
        if (sc.owner != uint32_t(a.n_tokens - n)) continue;   // one warp per tile
        const int kvh = int(t % a.hkv);
        const float so_k = a.k_scales[t], so_v = a.v_scales[t];
        // sc.rows holds at least this warp's own row
        const int r0 = __ffs(sc.rows) - 1;
        const long long src0 = ((long long)a.row_tok[t * kBlockSize + r0] * a.hkv + kvh) * D;
        float xk[EPL], xv[EPL];
        load_row<S, D>(a.k_new, src0, xk);
        load_row<S, D>(a.v_new, src0, xv);
        bool grow_k, grow_v;
        const float sk = settle_scale(sc.amax_k, so_k, &grow_k);
        const float sv = settle_scale(sc.amax_v, so_v, &grow_v);
        if (grow_k) requant_tile<D>(a.k_cache + t * kBlockSize * D, so_k, sk, lane);
        if (grow_v) requant_tile<D>(a.v_cache + t * kBlockSize * D, so_v, sv, lane);
        __syncwarp();
        const long long dst0 = (t * kBlockSize + r0) * D + lane * EPL;
        store_codes<EPL>(a.k_cache, dst0, xk, sk);
        store_codes<EPL>(a.v_cache, dst0, xv, sv);
        // the call's other new rows of the tile
        for (uint32_t m = sc.rows & (sc.rows - 1); m; m &= m - 1) {
            const int r = __ffs(m) - 1;
            const long long src = ((long long)a.row_tok[t * kBlockSize + r] * a.hkv + kvh) * D;
            load_row<S, D>(a.k_new, src, xk);
            load_row<S, D>(a.v_new, src, xv);
            const long long dst = (t * kBlockSize + r) * D + lane * EPL;
            store_codes<EPL>(a.k_cache, dst, xk, sk);
            store_codes<EPL>(a.v_cache, dst, xv, sv);
        }
        if (lane == 0) {
            a.k_scales[t] = sk;
            a.v_scales[t] = sv;
            *ts = TileScratch{0u, 0u, 0u, 0u};   // zero again for the next call
        }
    }
}

// The decode step's append over an INT8 cache: one new token per sequence,
// at position L_b - 1, so each (block, kv head) tile receives exactly one
// row and its warp needs no gather pass: the same settle, requantisation and
// encoding as i8_settle_kernel, for the one row (codes and scales come out
// bit for bit as pkv_append's for the same slots). One warp per (sequence,
// kv head); sequences with L = 0, an over-long length or an out-of-pool
// table entry write nothing (the split kernel flags them).
struct I8StepArgs {
    const void* k_new;            // [batch, hkv, D]
    const void* v_new;
    int8_t* k_cache;
    int8_t* v_cache;
    float* k_scales;
    float* v_scales;
    const int32_t* block_tables;  // [batch, mb]
    const int32_t* context_lens;
    uint32_t* status;
    int batch, hkv, mb, num_blocks;
};

template <typename S, int D>
__global__ void __launch_bounds__(kThreads, 4) i8_step_append_kernel(I8StepArgs a) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int EPL = D / 32;
    const int lane = threadIdx.x & 31;
    const long long items = (long long)a.batch * a.hkv;
    for (long long it = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; it < items;
         it += ((long long)gridDim.x * blockDim.x) >> 5) {
        const int b = int(it / a.hkv), kvh = int(it - (long long)b * a.hkv);
        // the new rows are loaded while the slot is resolved
        float xk[EPL], xv[EPL];
        load_row<S, D>(a.k_new, it * D, xk);
        load_row<S, D>(a.v_new, it * D, xv);
        const int L = a.context_lens[b];
        if (L <= 0 || L > a.mb * kBlockSize) continue;
        const int blk = a.block_tables[(long long)b * a.mb + (L - 1) / kBlockSize];
        if (unsigned(blk) >= unsigned(a.num_blocks)) continue;
        const long long t = (long long)blk * a.hkv + kvh;
        const int r = (L - 1) % kBlockSize;
        const float so_k = a.k_scales[t], so_v = a.v_scales[t];
        float mk = 0.f, mv = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            mk = fmaxf(mk, fabsf(xk[e]));
            mv = fmaxf(mv, fabsf(xv[e]));
        }
        mk = warp_max(mk);
        mv = warp_max(mv);
        bool grow_k, grow_v;
        const float sk = settle_scale(__float_as_uint(mk), so_k, &grow_k);
        const float sv = settle_scale(__float_as_uint(mv), so_v, &grow_v);
        if (grow_k) requant_tile<D>(a.k_cache + t * kBlockSize * D, so_k, sk, lane);
        if (grow_v) requant_tile<D>(a.v_cache + t * kBlockSize * D, so_v, sv, lane);
        __syncwarp();
        const long long dst = (t * kBlockSize + r) * D + lane * EPL;
        store_codes<EPL>(a.k_cache, dst, xk, sk);
        store_codes<EPL>(a.v_cache, dst, xv, sv);
        if (lane == 0) {
            a.k_scales[t] = sk;
            a.v_scales[t] = sv;
        }
    }
}

int grid_for(long long work_items, int per_block, int cap) {
    long long g = (work_items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    return int(g < cap ? g : cap);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

pkv_status check_cache(const pkv_cache_desc* c) {
    if (!c) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return PKV_ERR_INVALID_ARG;
    if (c->kv_dtype != PKV_F16 && c->kv_dtype != PKV_BF16 && c->kv_dtype != PKV_I8)
        return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

template <typename S, int D>
void launch_i8(const I8Args& a, cudaStream_t st) {
    const long long items = (long long)a.n_tokens * a.hkv;
    const int g = grid_for(items, kWarps, 1 << 16);
    launch_pdl(i8_gather_kernel<S, D>, dim3(g), dim3(kThreads), 0, st, a);
    launch_pdl(i8_settle_kernel<S, D>, dim3(g), dim3(kThreads), 0, st, a);
}

template <typename S, int D>
cudaError_t launch_i8_step(const I8StepArgs& a, cudaStream_t st) {
    const long long items = (long long)a.batch * a.hkv;
    return launch_pdl(i8_step_append_kernel<S, D>, dim3(grid_for(items, kWarps, 1 << 16)),
                      dim3(kThreads), 0, st, a);
}

}  // namespace

// The INT8 decode step's append (see i8_step_append_kernel); the caller has
// checked the arguments.
cudaError_t launch_i8_step_append(const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                  void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                  const int32_t* block_tables, int mb, const int32_t* context_lens,
                                  int batch, int hkv, int D, int num_blocks, uint32_t* status,
                                  cudaStream_t stream) {
    I8StepArgs a;
    a.k_new = k_new; a.v_new = v_new;
    a.k_cache = static_cast<int8_t*>(k_cache); a.v_cache = static_cast<int8_t*>(v_cache);
    a.k_scales = k_scales; a.v_scales = v_scales;
    a.block_tables = block_tables; a.context_lens = context_lens; a.status = status;
    a.batch = batch; a.hkv = hkv; a.mb = mb; a.num_blocks = num_blocks;
    if (src_dtype == PKV_BF16)
        return D == 128 ? launch_i8_step<BF16, 128>(a, stream) : launch_i8_step<BF16, 64>(a, stream);
    return D == 128 ? launch_i8_step<F16, 128>(a, stream) : launch_i8_step<F16, 64>(a, stream);
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_append_workspace_size(const pkv_cache_desc* cache) {
    if (check_cache(cache) != PKV_OK) return 0;
    if (cache->kv_dtype != PKV_I8) return 0;
    const size_t tiles = size_t(cache->num_blocks) * size_t(cache->num_kv_heads);
    return tiles * (sizeof(TileScratch) + kBlockSize * sizeof(int32_t));
}

extern "C" pkv_status pkv_append(const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                 int32_t num_tokens, const int64_t* slot_mapping, void* k_cache,
                                 void* v_cache, float* k_scales, float* v_scales,
                                 const pkv_cache_desc* cache, void* workspace,
                                 size_t workspace_bytes, uint32_t* dev_status,
                                 cudaStream_t stream) {
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    if (dev_status && !aligned(dev_status, 4)) return PKV_ERR_INVALID_ARG;
    const int D = cache->head_dim, hkv = cache->num_kv_heads;
    const long long pool_slots = (long long)cache->num_blocks * kBlockSize;

    if (cache->kv_dtype != PKV_I8) {
        if (src_dtype != cache->kv_dtype) return PKV_ERR_INVALID_ARG;
        const int vpr = D * 2 / 16;
        const long long total = (long long)num_tokens * hkv * vpr;
        launch_pdl(append_copy_kernel, dim3(grid_for(total, kThreads, 152 * 32)), dim3(kThreads),
                   0, stream, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                   slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                   num_tokens, hkv, vpr, pool_slots, dev_status);
    } else {
        if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
        if (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4))
            return PKV_ERR_INVALID_ARG;
        const size_t need = pkv_append_workspace_size(cache);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return PKV_ERR_WORKSPACE;
        const size_t tiles = size_t(cache->num_blocks) * size_t(hkv);
        TileScratch* ws = static_cast<TileScratch*>(workspace);
        I8Args a{k_new, v_new, slot_mapping, static_cast<int8_t*>(k_cache),
                 static_cast<int8_t*>(v_cache), k_scales, v_scales, ws,
                 reinterpret_cast<int32_t*>(ws + tiles), dev_status, num_tokens, hkv, pool_slots};
        if (src_dtype == PKV_BF16) {
            if (D == 128) launch_i8<BF16, 128>(a, stream); else launch_i8<BF16, 64>(a, stream);
        } else {
            if (D == 128) launch_i8<F16, 128>(a, stream); else launch_i8<F16, 64>(a, stream);
        }
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: bad pointer, size or shape";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: configuration not built";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing or too small";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA: CUDA call or launch failed";
    }
    return "PKV_ERR_UNKNOWN";
}
