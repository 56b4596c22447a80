// Paged decode attention: split kernel (stream of KV blocks per worker warp)
// and combine kernel (split-K reduce of partial softmax states).
//
// The method: one query token per sequence attends over its context, whose
// K/V sit in fixed-size physical blocks reached through the sequence's block
// table; the kernel gathers the blocks itself, with no compaction copy
// (Continuous-Batching-LLM-Inference-Engine README, feature list "Paged
// KV-cache", "PagedAttention kernel"; mini-inference-engine component "Paged
// decode attention"; paged-inference-engine overview, "paged INT8 KV
// storage").
//
// GB300 design:
// * Work is the stream of units (sequence b, kv head, block j), ordered
//   b-major, then kv head, then j, so each (b, kv head) "segment" is
//   contiguous. The stream is cut into W equal ranges, one per worker warp:
//   every warp moves the same number of bytes whatever the length mix.
// * Each warp owns a ring of stages in shared memory. Lane 0 issues one bulk
//   (TMA) copy for the 16-row K tile and one for the V tile of a unit (each a
//   contiguous run of the cache), completing on the stage's mbarrier; INT8
//   scales follow by cp.async on the same barrier. Block-table entries for the
//   next 32 units are fetched ahead, one per lane.
// * All g query heads of a KV head are served by the warp that reads its
//   tiles, so each tile is read from HBM once. Both contractions run on the
//   tensor cores (mma.sync m16n8k16, fp32 accumulators): scores as
//   S[16 tokens x 8 head columns] (g <= 8 heads, padded), P.V as
//   O^T[dims x heads] += V^T[dims x 16 tokens] P^T, so each lane keeps the
//   online-softmax state (running max and sum, exp2 domain) of its own two
//   heads. INT8 codes enter the MMAs as exact fp16 values with a bias that is
//   taken off per head.
// * A segment that lies inside one warp's range is normalised and written
//   out directly. Pieces of a segment that crosses ranges leave (m, l, o) in
//   the workspace at slot (segment + worker), which is unique because both
//   partitions are contiguous in the same order; the combine kernel merges
//   them.
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kMaxWarpsPerCta = 8;   // scan scratch slots at the start of shared memory
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 100 ms when draining
constexpr int kMaxBatch = 8192;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// a if c else b, per 32-bit word (lane-dependent register selection)
__device__ __forceinline__ uint4 sel4(bool c, const uint4& a, const uint4& b) {
    return make_uint4(c ? a.x : b.x, c ? a.y : b.y, c ? a.z : b.z, c ? a.w : b.w);
}

// The block prefix kept in shared memory has at most kPrefixEntries + 1
// entries, so that its size does not grow with the batch: up to
// kPrefixEntries sequences it is exact (stride 1); beyond, it holds every
// stride-th entry, stride = ceil(batch / kPrefixEntries), and a lookup ends
// with a scan of at most stride context lengths.
constexpr int kPrefixEntries = 256;
// Largest shared-memory prefix area (scan scratch + prefix), any batch.
constexpr int kPrefixMaxBytes = align_up(4 * kMaxWarpsPerCta + 4 * (kPrefixEntries + 1), 128);

template <typename KV, int D, int G>
struct Cfg {
    static constexpr int esize = Elem<KV>::bytes;
    static constexpr int kI8 = (esize == 1);
    // Blocks per work unit: 2 for INT8 caches (a unit of 32 tokens halves the
    // per-token share of the softmax bookkeeping, the waits and the copy
    // issue, which bound the INT8 kernel), 1 for 16-bit caches.
    static constexpr int UB = kI8 ? 2 : 1;
    static constexpr int UT = UB * kBlockSize;                    // tokens per unit
    static constexpr int TILE = kBlockSize * D * esize;          // bytes of one K (or V) tile
    static constexpr int ROW = D * esize;                         // bytes of one token row
    static constexpr int STAGE = 2 * UB * TILE;                   // K tiles [UB], V tiles [UB]
    // Stages per warp: as many as fit ~19 KB per warp with their q slots, so
    // that 3 CTAs of 4 warps share an SM (at least 2 stages).
    static constexpr int QBYTES = G * D * 2;   // q rows of one (sequence, kv head)
    static constexpr int NS = (19456 / (STAGE + QBYTES)) < 2 ? 2 : (19456 / (STAGE + QBYTES));
    // Per-warp shared-memory region.
    static constexpr int OFF_BAR = NS * STAGE;                       // 8-byte mbarriers
    static constexpr int OFF_META = align_up(OFF_BAR + NS * 8, 16);   // int4 per stage
    static constexpr int OFF_SCL = OFF_META + NS * 16;                // float2 per stage, block
    static constexpr int OFF_P = align_up(OFF_SCL + NS * UB * 8, 16); // float4 reads
    // P[head][token] rows in shared memory: UT floats each (INT8: UT fp16
    // values, the B operand's type, in the same space)
    static constexpr int PS = UT;
    // q rows of a piece's (sequence, kv head), copied with its first unit
    static constexpr int OFF_Q = align_up(OFF_P + PS * G * 4, 128);
    static constexpr int WARP_BYTES = align_up(OFF_Q + NS * QBYTES, 128);
    // Worker warps per CTA: 4 (three CTAs share an SM); INT8 units take more
    // shared memory than three 4-warp CTAs can have, so INT8 runs CTAs of 6
    // warps, two per SM (228 KB of shared memory, 1 KB reserved per CTA, and
    // the block prefix, at most kPrefixMaxBytes at any batch), which keeps 12
    // warps per SM.
    static constexpr int kSmemPerSm = 233472, kReservedPerCta = 1024;
    static constexpr int WARPS =
        (kI8 && 2 * (6 * WARP_BYTES + kPrefixMaxBytes + kReservedPerCta) <= kSmemPerSm) ? 6 : 4;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int MIN_CTAS = WARPS == 6 ? 2 : 3;   // launch bounds: registers per thread
    static_assert(NS >= 2 && NS <= 32, "stage count (one parity bit per stage)");
    static_assert(STAGE % 128 == 0 && OFF_Q % 128 == 0 && QBYTES % 16 == 0, "copy alignment");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size (heads fill <= 8 MMA columns)");
};

__host__ __device__ inline int prefix_stride(int batch) {
    return batch <= kPrefixEntries ? 1 : (batch + kPrefixEntries - 1) / kPrefixEntries;
}
__host__ __device__ inline int prefix_chunks(int batch) {
    const int st = prefix_stride(batch);
    return (batch + st - 1) / st;
}
// Dynamic shared memory starts with kMaxWarpsPerCta ints of scan scratch, then
// the block prefix [chunks + 1]; the per-warp regions follow, 128-byte aligned.
__host__ __device__ inline int prefix_bytes(int batch) {
    return align_up(4 * kMaxWarpsPerCta + 4 * (prefix_chunks(batch) + 1), 128);
}

// Workers that get units: at most one per kMinUnits units, so every range is
// non-empty and short batches are not cut into single-block pieces. The split
// and combine kernels derive it from the same U and agree on it.
constexpr long long kMinUnits = 4;
__host__ __device__ inline long long eff_workers(long long U, long long W) {
    const long long cap = U / kMinUnits;
    return cap < 1 ? 1 : (cap < W ? cap : W);
}

struct DecodeParams {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const float* k_scales;
    const float* v_scales;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    float* part_o;        // [slots, G, D]
    float* part_ml;       // [slots, G, 2]
    int32_t* ws_prefix;   // [batch + 1] copy of the block prefix for the combine
    uint32_t* status;
    const void* k_new;    // fused decode step: [batch, hkv, D] rows for position L - 1
    const void* v_new;    // (nullptr: attention only)
    int batch, hq, hkv, mb, num_blocks, workers;
    float qscale;         // softmax_scale * log2(e)
    uint64_t wait_ns;     // limit of each bounded wait on a stage (kWaitLimitNs)
    int stall_worker;     // test hook: this worker's first stage expects 16 bytes no
                          // copy delivers, so its wait runs out (-1: none)
};

__device__ __forceinline__ int clamp_len(int L, int mb, uint32_t* status, bool flag) {
    if (L < 0 || L > mb * kBlockSize) {
        if (flag) flag_status(status, PKV_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : mb * kBlockSize;
    }
    return L;
}

// Units (UT tokens each) of sequence b, from its clamped length.
template <int UT>
__device__ __forceinline__ int seq_units(const DecodeParams& p, int b) {
    return (clamp_len(__ldg(p.context_lens + b), p.mb, p.status, false) + UT - 1) / UT;
}

// Block prefix P[b] = sum_{b' < b} ceil(L_b' / UT) for b in [0, batch], UT =
// tokens per unit (16 UB); all threads. Shared memory keeps prefix[c] =
// P[c * stride] for c in [0, chunks) and prefix[chunks] = P[batch]; CTA 0
// writes the whole of P to ws_prefix for the combine.
template <int UT, int NT>
__device__ void build_prefix(const DecodeParams& p, int* warp_tot, int* prefix) {
    const int t = threadIdx.x;
    const int chunk = (p.batch + NT - 1) / NT;
    const int lo = min(p.batch, t * chunk), hi = min(p.batch, lo + chunk);
    const bool flag = blockIdx.x == 0;
    int sum = 0;
    for (int i = lo; i < hi; ++i)
        sum += (clamp_len(p.context_lens[i], p.mb, p.status, flag) + UT - 1) / UT;
    // exclusive scan of per-thread sums across the CTA
    const int lane = t & 31, warp = t >> 5;
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + inc - sum;
    const int stride = prefix_stride(p.batch);
    if (stride == 1) {
        for (int i = lo; i < hi; ++i) {
            prefix[i] = run;
            run += (clamp_len(p.context_lens[i], p.mb, p.status, false) + UT - 1) / UT;
        }
        if (t == NT - 1) prefix[p.batch] = run;
        __syncthreads();
        if (blockIdx.x == 0)
            for (int i = t; i <= p.batch; i += NT) p.ws_prefix[i] = prefix[i];
        return;
    }
    for (int i = lo; i < hi; ++i) {
        if (i % stride == 0) prefix[i / stride] = run;
        if (blockIdx.x == 0) p.ws_prefix[i] = run;
        run += (clamp_len(p.context_lens[i], p.mb, p.status, false) + UT - 1) / UT;
    }
    if (t == NT - 1) {
        prefix[prefix_chunks(p.batch)] = run;
        if (blockIdx.x == 0) p.ws_prefix[p.batch] = run;
    }
    __syncthreads();
}

// Unit u -> (b, kv head, unit j of the segment, i.e. blocks UB j .. UB j + UB - 1):
// b is the last sequence whose first unit is <= u (it always has units, since
// u < U). A binary search finds the last prefix chunk starting at or before
// u; with a strided prefix the chunk's sequences are then walked in order.
template <int UT>
__device__ __forceinline__ void decode_unit(long long u, const int* prefix, const DecodeParams& p,
                                            int& b, int& kvh, int& j) {
    const int x = int(u / p.hkv);
    const int stride = prefix_stride(p.batch), chunks = prefix_chunks(p.batch);
    int lo = 0;
    static_assert(kPrefixEntries <= 256, "search width: lo reaches at most 255");
    for (int step = 1 << 7; step; step >>= 1)
        if (lo + step < chunks && prefix[lo + step] <= x) lo += step;
    int first = prefix[lo], nb;
    if (stride == 1) {
        b = lo;
        nb = prefix[lo + 1] - first;
    } else {
        b = lo * stride;
        const int last = min(b + stride, p.batch) - 1;
        nb = seq_units<UT>(p, b);
        while (b < last && x >= first + nb) {   // ends inside the chunk since x < prefix[lo + 1]
            first += nb;
            nb = seq_units<UT>(p, ++b);
        }
    }
    const int r = int(u - (long long)p.hkv * first);
    kvh = r / nb;
    j = r - kvh * nb;
}

template <typename QT, int DPL>
__device__ __forceinline__ void store_out(void* out, long long off, const float2* v, float s) {
    uint32_t w[DPL / 2];
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
        if constexpr (std::is_same<QT, BF16>::value) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[i].x * s, v[i].y * s);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        } else {
            __half2 h = __floats2half2_rn(v[i].x * s, v[i].y * s);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    uint16_t* dst = static_cast<uint16_t*>(out) + off;
    if constexpr (DPL % 8 == 0) {
#pragma unroll
        for (int i = 0; i < DPL / 8; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else if constexpr (DPL == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
}

template <typename KV, typename QT, int D, int G>
__global__ void __launch_bounds__(Cfg<KV, D, G>::THREADS, Cfg<KV, D, G>::MIN_CTAS)
decode_split_kernel(const DecodeParams p) {
    using C = Cfg<KV, D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    int* prefix = reinterpret_cast<int*>(smem) + kMaxWarpsPerCta;
    griddep_wait();                 // inputs may come from the previous grid
    griddep_launch_dependents();    // the combine may start launching
    build_prefix<C::UT, C::THREADS>(p, reinterpret_cast<int*>(smem), prefix);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * C::WARPS + warp;
    const long long U = (long long)prefix[prefix_chunks(p.batch)] * p.hkv;
    const long long W = eff_workers(U, p.workers);
    if (w >= W || U == 0) return;
    const long long u0 = w * U / W, u1 = (w + 1) * U / W;

    unsigned char* region = smem + prefix_bytes(p.batch) + warp * C::WARP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(region + C::OFF_BAR);
    int4* meta = reinterpret_cast<int4*>(region + C::OFF_META);
    float2* scl = reinterpret_cast<float2*>(region + C::OFF_SCL);
    float* pbuf = reinterpret_cast<float*>(region + C::OFF_P);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < C::NS; ++s) mbar_init(smem_addr(&bars[s]), C::kI8 ? 2 : 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: block-table entries for 32 units at a time, one per lane
    // (blk1: the unit's second block for two-block units, while the sequence
    // reaches it)
    auto fetch = [&](long long base, int& b, int& kvh, int& j, int& blk, int& blk1, int& len) {
        const long long u = base + lane;
        blk1 = -1;
        if (u < u1) {
            decode_unit<C::UT>(u, prefix, p, b, kvh, j);
            const int32_t* row = p.block_tables + (long long)b * p.mb + C::UB * j;
            blk = __ldg(row);
            len = clamp_len(__ldg(p.context_lens + b), p.mb, p.status, false);
            if constexpr (C::UB == 2)
                if ((2 * j + 1) * kBlockSize < len) blk1 = __ldg(row + 1);
        } else {
            b = 0; kvh = 0; j = 0; blk = -1; len = 0;
        }
    };
    long long cbase = u0;
    int cb, ckvh, cj, cblk, cblk1, clen, xb, xkvh, xj, xblk, xblk1, xlen;
    fetch(cbase, cb, ckvh, cj, cblk, cblk1, clen);
    fetch(cbase + 32, xb, xkvh, xj, xblk, xblk1, xlen);

    auto issue = [&](long long u, int s, uint32_t extra_tx) {
        int idx = int(u - cbase);
        if (idx >= 32) {
            cbase += 32;
            cb = xb; ckvh = xkvh; cj = xj; cblk = xblk; cblk1 = xblk1; clen = xlen;
            fetch(cbase + 32, xb, xkvh, xj, xblk, xblk1, xlen);
            idx -= 32;
        }
        const int b = __shfl_sync(kFull, cb, idx);
        const int kvh = __shfl_sync(kFull, ckvh, idx);
        const int j = __shfl_sync(kFull, cj, idx);
        const int blk = __shfl_sync(kFull, cblk, idx);
        const int blk1 = (C::UB == 2) ? __shfl_sync(kFull, cblk1, idx) : -1;
        const int len = __shfl_sync(kFull, clen, idx);
        if (C::UB == 2 && lane == 0) {
            // Two-block unit (INT8): blocks 2j and 2j + 1, the second while the
            // sequence reaches it. K tiles at stage + i TILE, V tiles at stage +
            // (2 + i) TILE, block i's scales in scl[2 s + i]; meta flag bits:
            // 0 = block 0 copied, 1 = first unit of a piece, 3 = block 1 copied.
            const uint32_t bar = smem_addr(&bars[s]);
            const bool ok0 = unsigned(blk) < unsigned(p.num_blocks);
            const bool has1 = (2 * j + 1) * kBlockSize < len;
            const bool ok1 = has1 && unsigned(blk1) < unsigned(p.num_blocks);
            const bool first = (u == u0) || (j == 0);
            meta[s] = make_int4(b, kvh | ((ok0 ? 1 : 0) << 16) | ((first ? 1 : 0) << 17) |
                                       ((ok1 ? 1 : 0) << 19), j, len);
            const uint32_t tx = (ok0 ? 2 * C::TILE : 0) + (ok1 ? 2 * C::TILE : 0) +
                                (first ? C::QBYTES : 0) + extra_tx;
            if (tx) mbar_arrive_expect_tx(bar, tx);
            else mbar_arrive(bar);
            if (first)
                bulk_g2s(smem_addr(region + C::OFF_Q + s * C::QBYTES),
                         static_cast<const uint16_t*>(p.q) + ((long long)b * p.hq + kvh * G) * D,
                         C::QBYTES, bar);
            unsigned char* st = region + s * C::STAGE;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (!(i ? ok1 : ok0)) continue;
                const long long tile = (long long)(i ? blk1 : blk) * p.hkv + kvh;
                bulk_g2s(smem_addr(st + i * C::TILE),
                         static_cast<const char*>(p.k_cache) + tile * C::TILE, C::TILE, bar);
                bulk_g2s(smem_addr(st + (2 + i) * C::TILE),
                         static_cast<const char*>(p.v_cache) + tile * C::TILE, C::TILE, bar);
                cp_async_4(smem_addr(&scl[2 * s + i].x), p.k_scales + tile);
                cp_async_4(smem_addr(&scl[2 * s + i].y), p.v_scales + tile);
            }
            if (ok0 || ok1) cp_async_arrive_noinc(bar);
            else mbar_arrive(bar);
            if (!ok0 || (has1 && !ok1)) flag_status(p.status, PKV_DEV_BAD_BLOCK);
        } else if (C::UB == 1 && lane == 0) {
            const uint32_t bar = smem_addr(&bars[s]);
            const bool ok = unsigned(blk) < unsigned(p.num_blocks);
            const bool first = (u == u0) || (j == 0);   // first unit of a piece
            // Fused decode step: the tile holding the sequence's new token
            // (position len - 1, row r) takes rows [0, r) from the cache and
            // row r from k_new / v_new; the consumer then stores row r into
            // the cache. Rows past r are masked, so they are not copied.
            const bool fuse = !C::kI8 && ok && p.k_new != nullptr && len > 0 &&
                              j == (len - 1) / kBlockSize &&
                              __ldg(p.context_lens + b) == len;   // not clamped: flagged, no write
            const int r = fuse ? (len - 1) % kBlockSize : kBlockSize;
            meta[s] = make_int4(b, kvh | ((ok ? 1 : 0) << 16) | ((first ? 1 : 0) << 17) |
                                       ((fuse ? 1 : 0) << 18), j, len);
            if (fuse) scl[s].x = __int_as_float(blk);   // scales are unused for 16-bit caches
            const uint32_t tx = (ok ? 2 * (fuse ? (r + 1) * C::ROW : C::TILE) : 0) +
                                (first ? C::QBYTES : 0) + extra_tx;
            if (tx) mbar_arrive_expect_tx(bar, tx);
            else mbar_arrive(bar);
            if (first)
                bulk_g2s(smem_addr(region + C::OFF_Q + s * C::QBYTES),
                         static_cast<const uint16_t*>(p.q) + ((long long)b * p.hq + kvh * G) * D,
                         C::QBYTES, bar);
            if (ok) {
                const long long tile = (long long)blk * p.hkv + kvh;
                unsigned char* st = region + s * C::STAGE;
                if (r > 0) {
                    bulk_g2s(smem_addr(st), static_cast<const char*>(p.k_cache) + tile * C::TILE,
                             r * C::ROW, bar);
                    bulk_g2s(smem_addr(st + C::TILE),
                             static_cast<const char*>(p.v_cache) + tile * C::TILE, r * C::ROW, bar);
                }
                if (fuse) {
                    const long long src = ((long long)b * p.hkv + kvh) * C::ROW;
                    bulk_g2s(smem_addr(st + r * C::ROW), static_cast<const char*>(p.k_new) + src,
                             C::ROW, bar);
                    bulk_g2s(smem_addr(st + C::TILE + r * C::ROW),
                             static_cast<const char*>(p.v_new) + src, C::ROW, bar);
                }
                if constexpr (C::kI8) {
                    cp_async_4(smem_addr(&scl[s].x), p.k_scales + tile);
                    cp_async_4(smem_addr(&scl[s].y), p.v_scales + tile);
                    cp_async_arrive_noinc(bar);
                }
            } else {
                flag_status(p.status, PKV_DEV_BAD_BLOCK);
                if constexpr (C::kI8) mbar_arrive(bar);
            }
        }
    };

    // ---- consumer: scores and P.V on the tensor cores (mma.sync m16n8k16,
    // fp32 accumulators), all cache types alike:
    //  * S[16 tokens x heads]: rows = the tile's tokens, columns = the g heads
    //    (padded to 8). Lane (gq, tq) = (lane / 4, lane % 4) then holds tokens
    //    gq and gq + 8 of heads 2tq and 2tq + 1.
    //  * O^T[dims x heads] += V^T[dims x 16 tokens] P^T[16 tokens x heads]: lane
    //    (gq, tq) accumulates dims [gq*D/8, (gq+1)*D/8) of heads 2tq, 2tq + 1,
    //    so its softmax state is that of its own two heads.
    // 16-bit caches multiply in their own type. INT8 codes c enter as the
    // fp16 value 1152 + c, exact (the byte c + 128 as the low mantissa byte of
    // 1024): the bias adds 1152 * sum_d q_d to every score of a head, taken
    // off before the block's K scale, and 1152 * sum_t P_t to every O entry
    // of a head, taken off when the piece is written (sum_t P_t kept beside
    // O with the same rescalings). q is rounded to fp16 and the block's V
    // scale rides on P.
    using MMT = typename std::conditional<C::kI8, F16, KV>::type;   // mma operand type
    constexpr int MT = D / 16;                   // m-tiles of P.V
    constexpr int DL = D / 8;                    // dims a lane row group owns
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t qb[D / 16][2];                      // B fragments of q, per k-step
    float m[2], lsum[2] = {0.f, 0.f};            // heads 2tq, 2tq + 1
    float oa[MT][4];                             // O^T accumulators
    int pb = -1, pkvh = -1, first_j = 0, last_j = 0, plen = 0;
    // INT8: P carries the block's V scale into fp16, so O is kept in units of
    // 2^vexp (vexp >= 0, raised when a scale would push P past 2^14, i.e.
    // toward the fp16 limit) and multiplied back when the piece is written.
    int vexp = 0;
    float vmul = 1.f;                            // 2^-vexp
    float kbias[2] = {0.f, 0.f};                 // INT8: 1152 * sum_d q_d, heads 2tq + e
    float pv[2] = {0.f, 0.f};                    // INT8: sum_t P_t of this lane's tokens

    auto finalize = [&]() {
        const int nbk = (plen + C::UT - 1) / C::UT;   // plen: pb's clamped length
        const long long seg = (long long)pb * p.hkv + pkvh;
        const bool whole = (first_j == 0 && last_j == nbk - 1);
        float lh[2] = {lsum[0], lsum[1]};
        float ph[2] = {pv[0], pv[1]};
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                lh[e] += __shfl_xor_sync(kFull, lh[e], off);
                if constexpr (C::kI8) ph[e] += __shfl_xor_sync(kFull, ph[e], off);
            }
        const float up = C::kI8 ? ldexpf(1.f, vexp) : 1.f;   // O back from units of 2^vexp
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tq + e;
            if (h >= G) continue;
            if constexpr (C::kI8) {   // the V bias: O -= 1152 * sum_t P_t
                const float cb = 1152.f * ph[e];
#pragma unroll
                for (int i = 0; i < MT; ++i) { oa[i][e] -= cb; oa[i][2 + e] -= cb; }
            }
            if (whole) {
                float2 v[MT];
#pragma unroll
                for (int i = 0; i < MT; ++i) v[i] = make_float2(oa[i][e], oa[i][2 + e]);
                const float inv = lh[e] > 0.f ? up / lh[e] : 0.f;
                store_out<QT, DL>(p.out, ((long long)pb * p.hq + pkvh * G + h) * D + gq * DL, v, inv);
            } else {
                const long long slot = seg + w;
                float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * G + h) * D + gq * DL);
#pragma unroll
                for (int i = 0; i < MT / 2; ++i)
                    dst[i] = make_float4(oa[2 * i][e] * up, oa[2 * i][2 + e] * up,
                                         oa[2 * i + 1][e] * up, oa[2 * i + 1][2 + e] * up);
                if (gq == 0)
                    *reinterpret_cast<float2*>(p.part_ml + (slot * G + h) * 2) = make_float2(m[e], lh[e]);
            }
        }
    };

    // A fragments of V^T for m-tile i: rows gq, gq + 8 = dims gq*DL + 2i, + 1;
    // columns = tokens 2tq, 2tq + 1 (a0, a1) and 2tq + 8, 2tq + 9 (a2, a3).
    // Tokens at or past `nv` are zeroed (stale rows may hold anything, and
    // 0 * NaN would poison the sum).
    uint32_t va[MT][4];
    // The V data of the lane's four rows, read before the softmax (its P
    // stores would otherwise order these shared-memory reads after them).
    // 16-bit: lanes of odd tq read a row's two 16-byte chunks in the other
    // order (halves the bank conflicts of rows that share the bank mapping).
    uint4 vx16[4][C::kI8 ? 1 : DL / 8];
    auto read_v16 = [&](const unsigned char* vt) {
        const int vswap = (DL / 8 == 2) ? (tq & 1) : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 2 * tq + (i & 1) + 8 * (i >> 1);
            const unsigned char* row = vt + t * C::ROW + gq * DL * 2;
#pragma unroll
            for (int c = 0; c < DL / 8; ++c)
                vx16[i][c] = *reinterpret_cast<const uint4*>(row + 16 * (c ^ vswap));
        }
    };
    uint32_t vw8[C::UB][4][C::kI8 ? DL / 4 : 1];   // INT8: per block of the unit
    auto read_v8 = [&](const unsigned char* vt, int blk_i) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 2 * tq + (i & 1) + 8 * (i >> 1);
            const unsigned char* row = vt + t * C::ROW + gq * DL;
            if constexpr (DL == 16) {
                const uint4 x = *reinterpret_cast<const uint4*>(row);
                vw8[blk_i][i][0] = x.x; vw8[blk_i][i][1] = x.y;
                vw8[blk_i][i][2] = x.z; vw8[blk_i][i][3] = x.w;
            } else if constexpr (DL == 8) {
                const uint2 x = *reinterpret_cast<const uint2*>(row);
                vw8[blk_i][i][0] = x.x; vw8[blk_i][i][1] = x.y;
            }
        }
    };
    auto load_v = [&](const unsigned char* vt, int nv, int blk_i) {
        if constexpr (!C::kI8) {
            // 16-bit: DL dims of each of the lane's four rows (read by read_v16)
            (void)vt;
            (void)blk_i;
            uint32_t vw[4][DL / 2];
            const int vswap = (DL / 8 == 2) ? (tq & 1) : 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 2 * tq + (i & 1) + 8 * (i >> 1);
                const uint4* x = vx16[i];
                const bool keep = t < nv;
#pragma unroll
                for (int c = 0; c < DL / 8; ++c) {
                    uint4 v = (DL / 8 == 2) ? sel4(vswap != 0, x[(c ^ 1) & (DL / 8 - 1)], x[c]) : x[c];
                    if (!keep) v = make_uint4(0u, 0u, 0u, 0u);
                    vw[i][4 * c] = v.x; vw[i][4 * c + 1] = v.y;
                    vw[i][4 * c + 2] = v.z; vw[i][4 * c + 3] = v.w;
                }
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                va[i][0] = __byte_perm(vw[0][i], vw[1][i], 0x5410);
                va[i][1] = __byte_perm(vw[0][i], vw[1][i], 0x7632);
                va[i][2] = __byte_perm(vw[2][i], vw[3][i], 0x5410);
                va[i][3] = __byte_perm(vw[2][i], vw[3][i], 0x7632);
            }
        } else {
            // INT8: DL codes per row (read by read_v8); the bytes of two
            // tokens are interleaved, then each pair becomes the fp16x2
            // (1152 + c0, 1152 + c1). Rows past the context need no zeroing:
            // any byte is a finite code and its P is exactly 0.
            (void)vt;
            (void)nv;
            auto& vw = vw8[blk_i];
#pragma unroll
            for (int k = 0; k < DL / 4; ++k) {
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {   // bytes 0-1 -> m-tile 2k, bytes 2-3 -> 2k + 1
                    const uint32_t sel = hb ? 0x7362u : 0x5140u;
                    const uint32_t x = __byte_perm(vw[0][k], vw[1][k], sel) ^ 0x80808080u;
                    const uint32_t y = __byte_perm(vw[2][k], vw[3][k], sel) ^ 0x80808080u;
                    const int i = 2 * k + hb;
                    va[i][0] = i8x2_biased_h2(x, 0x4140);
                    va[i][1] = i8x2_biased_h2(x, 0x4342);
                    va[i][2] = i8x2_biased_h2(y, 0x4140);
                    va[i][3] = i8x2_biased_h2(y, 0x4342);
                }
            }
        }
    };

    for (int s = 0; s < C::NS; ++s)
        if (u0 + s < u1) issue(u0 + s, s, (s == 0 && w == p.stall_worker) ? 16u : 0u);
    long long u_issue = (u0 + C::NS < u1) ? u0 + C::NS : u1;
    uint32_t parity = 0;
    long long u = u0;
    bool aborted = false;
    int s = 0;                       // stage of unit u
    for (; u < u1; ++u, s = (s + 1 == C::NS) ? 0 : s + 1) {
        const uint32_t bar = smem_addr(&bars[s]);
        const bool got = mbar_wait_bounded(bar, (parity >> s) & 1u, p.wait_ns);
        if (!__all_sync(kFull, got)) {
            if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
            aborted = true;
            break;
        }
        parity ^= 1u << s;
        const int4 mt = meta[s];
        const int flags = mt.y >> 16;
        if (flags & 2) {  // first unit of a new piece: its q rows came with it
            if (pb >= 0) finalize();
            pb = mt.x;
            pkvh = mt.y & 0xffff;
            first_j = mt.z;
            plen = mt.w;
            const unsigned char* qs = region + C::OFF_Q + s * C::QBYTES;
            // q^T as the B operand, with the contraction index permuted so that
            // one 16-byte load of a K row serves several k-steps. 16-bit: k-steps
            // 2c and 2c + 1 of lane tq read dims 32c + 8tq + [0, 4) and + [4, 8).
            // INT8: k-step kk of lane tq reads dims 16tq + 4(kk%4) + 64(kk/4) + [0, 4).
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if constexpr (!C::kI8) {
                    uint4 y = make_uint4(0u, 0u, 0u, 0u);
                    if (gq < G) y = *reinterpret_cast<const uint4*>(qs + 2 * (gq * D + 32 * c + 8 * tq));
                    qb[2 * c][0] = y.x; qb[2 * c][1] = y.y;
                    qb[2 * c + 1][0] = y.z; qb[2 * c + 1][1] = y.w;
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = 2 * c + h;
                        qb[kk][0] = qb[kk][1] = 0u;
                        if (gq < G) {
                            const int d0 = 16 * tq + 4 * (kk % 4) + 64 * (kk / 4);
                            const uint2 x = *reinterpret_cast<const uint2*>(qs + 2 * (gq * D + d0));
                            const float2 f0 = unpack2(QT{}, x.x), f1 = unpack2(QT{}, x.y);
                            qb[kk][0] = pack2<F16>(f0.x, f0.y);
                            qb[kk][1] = pack2<F16>(f1.x, f1.y);
                        }
                    }
                }
            }
            if constexpr (C::kI8) {
                // sum of the fp16 q of head gq (the values the MMAs multiply),
                // over the lane's dims, then over the 4 lanes of the head
                float qsum = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const float2 a = unpack2(F16{}, qb[kk][0]), b = unpack2(F16{}, qb[kk][1]);
                    qsum += (a.x + a.y) + (b.x + b.y);
                }
                qsum += __shfl_xor_sync(kFull, qsum, 1);
                qsum += __shfl_xor_sync(kFull, qsum, 2);
#pragma unroll
                for (int e = 0; e < 2; ++e)   // head 2tq + e lives in lanes 4(2tq + e) + [0, 4)
                    kbias[e] = 1152.f * __shfl_sync(kFull, qsum, (8 * tq + 4 * e) & 31);
                pv[0] = pv[1] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) { m[e] = -INFINITY; lsum[e] = 0.f; }
#pragma unroll
            for (int i = 0; i < MT; ++i) oa[i][0] = oa[i][1] = oa[i][2] = oa[i][3] = 0.f;
            vexp = 0;
            vmul = 1.f;
        }
        last_j = mt.z;

        if (flags & (C::UB == 2 ? 9 : 1)) {
            const unsigned char* kt = region + s * C::STAGE;   // K tiles of the unit
            const unsigned char* vt = kt + C::UB * C::TILE;    // V tiles
            const int nv = min(C::UT, plen - C::UT * mt.z);     // valid tokens of the unit
            float ksc[C::UB], vsc[C::UB];
            bool okb[C::UB];                                    // block i was copied
#pragma unroll
            for (int i = 0; i < C::UB; ++i) {
                ksc[i] = 1.f;
                vsc[i] = 1.f;
                okb[i] = (C::UB == 1) || ((flags >> (i ? 3 : 0)) & 1);
            }
            // scores S[token][head] of block i: two accumulator chains (even /
            // odd k-steps). Rows are D * esize bytes apart, a multiple of 128,
            // so all rows share the bank mapping: lanes of odd gq read the two
            // k-step groups of a 128-byte span in the other order, which
            // spreads each quarter warp over all 32 banks, and the groups are
            // put back in registers.
            float acc[C::UB][2][4];
#pragma unroll
            for (int i = 0; i < C::UB; ++i)
#pragma unroll
                for (int c = 0; c < 2; ++c) acc[i][c][0] = acc[i][c][1] = acc[i][c][2] = acc[i][c][3] = 0.f;
            const bool kswap = !C::kI8 && (gq & 1) != 0;
            if constexpr (!C::kI8) {
                if (flags & 4) {   // fused step: the new token's row goes to the cache
                    const int r = (mt.w - 1) % kBlockSize;
                    const long long tile = (long long)__float_as_int(scl[s].x) * p.hkv + (mt.y & 0xffff);
                    const long long dst = (tile * C::TILE + r * C::ROW) / 4;
                    const uint32_t* ks = reinterpret_cast<const uint32_t*>(kt + r * C::ROW);
                    const uint32_t* vs = reinterpret_cast<const uint32_t*>(vt + r * C::ROW);
                    uint32_t* kd = static_cast<uint32_t*>(const_cast<void*>(p.k_cache)) + dst;
                    uint32_t* vd = static_cast<uint32_t*>(const_cast<void*>(p.v_cache)) + dst;
                    for (int wv = lane; wv < C::ROW / 4; wv += 32) {
                        kd[wv] = ks[wv];
                        vd[wv] = vs[wv];
                    }
                }
#pragma unroll
                for (int c2 = 0; c2 < D / 32; c2 += 2) {
                    uint4 y[2][2];   // [load h: pair c2 + (h ^ kswap)][row gq, gq + 8]
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int off = 64 * (c2 + (h ^ (kswap ? 1 : 0))) + 16 * tq;
                        y[h][0] = *reinterpret_cast<const uint4*>(kt + gq * C::ROW + off);
                        y[h][1] = *reinterpret_cast<const uint4*>(kt + (gq + 8) * C::ROW + off);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = c2 + h;
                        const uint4 x0 = sel4(kswap, y[h ^ 1][0], y[h][0]);
                        const uint4 x1 = sel4(kswap, y[h ^ 1][1], y[h][1]);
                        const uint32_t a0[4] = {x0.x, x1.x, x0.y, x1.y};
                        const uint32_t a1[4] = {x0.z, x1.z, x0.w, x1.w};
                        mma16816<KV>(acc[0][0], a0, qb[2 * c][0], qb[2 * c][1]);
                        mma16816<KV>(acc[0][1], a1, qb[2 * c + 1][0], qb[2 * c + 1][1]);
                    }
                }
                read_v16(vt);
            } else {
                // the blocks' scales (0 for a block that was not copied: its
                // tokens are masked and its P is 0)
                float vmax = 0.f;
#pragma unroll
                for (int i = 0; i < C::UB; ++i) {
                    const float2 sc = scl[C::UB * s + i];
                    ksc[i] = okb[i] ? sc.x : 0.f;
                    vsc[i] = okb[i] ? sc.y : 0.f;
                    vmax = fmaxf(vmax, vsc[i]);
                }
                if (vmax * vmul >= 16384.f) {   // warp-uniform; raise vexp, rescale O exactly
                    int ex;
                    frexpf(vmax, &ex);          // vmax < 2^ex
                    const int nexp = ex - 14;   // vmax * 2^-nexp < 2^14
                    const float r = ldexpf(1.f, vexp - nexp);
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        oa[i][0] *= r; oa[i][1] *= r; oa[i][2] *= r; oa[i][3] *= r;
                    }
                    pv[0] *= r; pv[1] *= r;
                    vexp = nexp;
                    vmul = ldexpf(1.f, -nexp);
                }
#pragma unroll
                for (int i = 0; i < C::UB; ++i) vsc[i] *= vmul;
                // the lane's 16-byte chunk of each half row holds 4 k-steps' columns
                constexpr int NC = D / 64;
#pragma unroll
                for (int bi = 0; bi < C::UB; ++bi) {
                    const unsigned char* kb = kt + bi * C::TILE;
                    uint4 y[NC][2];
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        y[c][0] = *reinterpret_cast<const uint4*>(kb + gq * C::ROW + 64 * c + 16 * tq);
                        y[c][1] = *reinterpret_cast<const uint4*>(kb + (gq + 8) * C::ROW + 64 * c + 16 * tq);
                    }
                    uint32_t w0[D / 16], w1[D / 16];
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        w0[4 * c] = y[c][0].x; w0[4 * c + 1] = y[c][0].y;
                        w0[4 * c + 2] = y[c][0].z; w0[4 * c + 3] = y[c][0].w;
                        w1[4 * c] = y[c][1].x; w1[4 * c + 1] = y[c][1].y;
                        w1[4 * c + 2] = y[c][1].z; w1[4 * c + 3] = y[c][1].w;
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t u0 = w0[kk] ^ 0x80808080u, u1 = w1[kk] ^ 0x80808080u;
                        mma_16816_f16(acc[bi][kk & 1], i8x2_biased_h2(u0, 0x4140),
                                      i8x2_biased_h2(u1, 0x4140), i8x2_biased_h2(u0, 0x4342),
                                      i8x2_biased_h2(u1, 0x4342), qb[kk][0], qb[kk][1]);
                    }
                }
#pragma unroll
                for (int bi = 0; bi < C::UB; ++bi) read_v8(vt + bi * C::TILE, bi);
            }
            float sv[C::UB][2][2];   // [block][token gq / gq + 8][head 2tq + e]
#pragma unroll
            for (int bi = 0; bi < C::UB; ++bi) {
                const float sk = p.qscale * ksc[bi];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool hv = 2 * tq + e < G && okb[bi];
                    float s0 = acc[bi][0][e] + acc[bi][1][e], s1 = acc[bi][0][2 + e] + acc[bi][1][2 + e];
                    if constexpr (C::kI8) {   // the K bias comes off before the scale
                        s0 -= kbias[e];
                        s1 -= kbias[e];
                    }
                    sv[bi][0][e] = (hv && kBlockSize * bi + gq < nv) ? s0 * sk : -INFINITY;
                    sv[bi][1][e] = (hv && kBlockSize * bi + gq + 8 < nv) ? s1 * sk : -INFINITY;
                }
            }
            float alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float bme = fmaxf(sv[0][0][e], sv[0][1][e]);   // max over the unit's tokens
#pragma unroll
                for (int bi = 1; bi < C::UB; ++bi) bme = fmaxf(bme, fmaxf(sv[bi][0][e], sv[bi][1][e]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) bme = fmaxf(bme, __shfl_xor_sync(kFull, bme, off));
                const float mn = fmaxf(m[e], bme);
                alpha[e] = (mn == -INFINITY) ? 1.f : fast_exp2(m[e] - mn);
                m[e] = mn;
                float ls = lsum[e] * alpha[e], wsum = 0.f;
#pragma unroll
                for (int bi = 0; bi < C::UB; ++bi) {
                    const float p0 = (sv[bi][0][e] == -INFINITY) ? 0.f : fast_exp2(sv[bi][0][e] - mn);
                    const float p1 = (sv[bi][1][e] == -INFINITY) ? 0.f : fast_exp2(sv[bi][1][e] - mn);
                    ls = ls + p0 + p1;
                    if constexpr (C::kI8) {
                        // P times the block's V scale, rounded to fp16 here, so that
                        // the bias sum uses exactly the weights the MMA multiplies;
                        // stored as fp16, the B operand's own type
                        const __half2 h = __floats2half2_rn(p0 * vsc[bi], p1 * vsc[bi]);
                        const float2 r = __half22float2(h);
                        wsum += r.x + r.y;
                        if (2 * tq + e < G) {   // P[head][token]
                            __half* ph16 = reinterpret_cast<__half*>(pbuf);
                            ph16[(2 * tq + e) * C::PS + kBlockSize * bi + gq] = __low2half(h);
                            ph16[(2 * tq + e) * C::PS + kBlockSize * bi + gq + 8] = __high2half(h);
                        }
                    } else if (2 * tq + e < G) {   // P[head][token]
                        pbuf[(2 * tq + e) * C::PS + kBlockSize * bi + gq] = p0;
                        pbuf[(2 * tq + e) * C::PS + kBlockSize * bi + gq + 8] = p1;
                    }
                }
                lsum[e] = ls;
                if constexpr (C::kI8) pv[e] = fmaf(pv[e], alpha[e], wsum);
            }
            if (__any_sync(kFull, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    oa[i][0] *= alpha[0]; oa[i][1] *= alpha[1];
                    oa[i][2] *= alpha[0]; oa[i][3] *= alpha[1];
                }
            }
            if constexpr (!C::kI8) load_v(vt, nv, 0);
            __syncwarp();
            // P^T as the B operand: column gq = head gq, tokens 2tq, 2tq + 1 | + 8
            // of each block. 16-bit caches: P = hi + lo in two parts of the
            // operand type (hi = rn(P), lo = rn(P - hi), the difference exact in
            // fp32), so a weight in [0, 1] is off by at most 2^-18 (bf16): with
            // one 16-bit P a two-token context would be off by up to 2^-9 |v|.
            // INT8: one fp16 part (already rounded above), off by at most 2^-11
            // of the weight, i.e. 2^-11 max|v| on the output, far inside the
            // INT8 bound.
#pragma unroll
            for (int bi = 0; bi < C::UB; ++bi) {
                if constexpr (C::kI8) load_v(vt, nv, bi);
                uint32_t ph[2] = {0u, 0u}, pl[2] = {0u, 0u};
                if (gq < G) {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        if constexpr (C::kI8) {   // two fp16 weights, tokens 2tq + 8k, + 1
                            ph[k] = *reinterpret_cast<const uint32_t*>(
                                reinterpret_cast<const __half*>(pbuf) + gq * C::PS +
                                kBlockSize * bi + 2 * tq + 8 * k);
                        } else {
                            const float2 f = *reinterpret_cast<const float2*>(
                                pbuf + gq * C::PS + kBlockSize * bi + 2 * tq + 8 * k);
                            ph[k] = pack2<MMT>(f.x, f.y);
                            const float2 r = unpack2(MMT{}, ph[k]);
                            pl[k] = pack2<MMT>(f.x - r.x, f.y - r.y);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) mma16816<MMT>(oa[i], va[i], ph[0], ph[1]);
                if constexpr (!C::kI8) {
#pragma unroll
                    for (int i = 0; i < MT; ++i) mma16816<MMT>(oa[i], va[i], pl[0], pl[1]);
                }
            }
        }
        // The stage goes back to the copy engine only after the math: releasing
        // it right after its reads (with V held in registers) measured slower.
        __syncwarp();
        if (u_issue < u1) {
            issue(u_issue, s, 0u);
            ++u_issue;
        }
    }
    if (!aborted) {
        if (pb >= 0) finalize();
        return;
    }
    // A copy never completed: give the others a short bounded wait, then leave.
    for (long long v = u; v < u_issue; ++v) {
        const int sv = int((v - u0) % C::NS);
        mbar_wait_bounded(smem_addr(&bars[sv]), (parity >> sv) & 1u, kDrainLimitNs);
        parity ^= 1u << sv;
    }
}

// ---------------------------------------------------------------- combine ---
struct CombineParams {
    const float* part_o;
    const float* part_ml;
    const int32_t* ws_prefix;
    void* out;
    int batch, hq, hkv, workers;
    int segs_per_cta;     // segments (sequence, kv head) each CTA looks after
};

// Worker whose range holds unit u: the largest w with floor(w*U/W) <= u.
__device__ __forceinline__ long long worker_of(long long u, long long U, long long W) {
    return ((u + 1) * W - 1) / U;
}

constexpr int kCombineThreads = 256;
// Resident combine CTAs per SM (a full SM of threads: at most 32 registers).
constexpr int kCombineCtasPerSm = 8;

// Fold one partial state (m, l, o) into a running merge (M, den, num), all in
// base 2: the running sums are rescaled when the maximum grows.
__device__ __forceinline__ void merge_state(float& M, float& den, float4& num, float m, float l,
                                            const float4& o) {
    if (m == -INFINITY) return;              // piece saw no valid token
    if (m > M) {
        const float r = (M == -INFINITY) ? 0.f : fast_exp2(M - m);
        den *= r;
        num.x *= r; num.y *= r; num.z *= r; num.w *= r;
        M = m;
    }
    const float a = fast_exp2(m - M);
    den += a * l;
    num.x += a * o.x; num.y += a * o.y; num.z += a * o.z; num.w += a * o.w;
}

// Merge the pieces wf..wl of segment seg (sequence b, kv head kvh):
// out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i (scores are in log2
// units). The CTA's threads form GROUPS groups of G*D/4 threads (one float4 of
// output each): group k merges pieces k, k + GROUPS, ... and the groups merge
// in shared memory. Every thread of the CTA calls it with the same segment.
template <typename QT, int D, int G>
__device__ __forceinline__ void merge_segment(const CombineParams& c, long long seg, int b, int kvh,
                                              int wf, int wl, float* s_m, float* s_den,
                                              float4* s_num) {
    constexpr int Q = D / 4, ITEMS = G * Q, GROUPS = kCombineThreads / ITEMS;
    const int t = threadIdx.x, item = t % ITEMS, grp = t / ITEMS;
    const int h = item / Q, d4 = item - h * Q;
    float M = -INFINITY, den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int w = wf + grp; w <= wl; w += GROUPS) {
        const long long slot = seg + w;
        const float2 ml = *reinterpret_cast<const float2*>(c.part_ml + (slot * G + h) * 2);
        const float4 o = *reinterpret_cast<const float4*>(c.part_o + (slot * G + h) * D + d4 * 4);
        merge_state(M, den, num, ml.x, ml.y, o);
    }
    if constexpr (GROUPS > 1) {
        s_m[t] = M;
        s_den[t] = den;
        s_num[t] = num;
        __syncthreads();
        if (grp == 0) {
#pragma unroll
            for (int k = 1; k < GROUPS; ++k) {
                const int o = k * ITEMS + item;
                // s_num holds unnormalised sums relative to s_m: merge as a state
                merge_state(M, den, num, s_m[o], s_den[o], s_num[o]);
            }
        }
    }
    if (grp == 0) {
        const long long obase = ((long long)b * c.hq + kvh * G + h) * D + d4 * 4;
        const float inv = den > 0.f ? 1.0f / den : 0.f;
        const float2 v[2] = {make_float2(num.x, num.y), make_float2(num.z, num.w)};
        store_out<QT, 4>(c.out, obase, v, inv);
    }
}

// Zero row for the empty sequence b, kv head kvh.
template <typename QT, int D, int G>
__device__ __forceinline__ void zero_segment(const CombineParams& c, int b, int kvh) {
    constexpr int Q = D / 4, ITEMS = G * Q;
    const int t = threadIdx.x, item = t % ITEMS;
    const int h = item / Q, d4 = item - h * Q;
    if (t < ITEMS) {
        const float2 z[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        store_out<QT, 4>(c.out, ((long long)b * c.hq + kvh * G + h) * D + d4 * 4, z, 0.f);
    }
}

// One CTA per segment (sequence b, kv head): write zeros for an empty
// sequence, merge the pieces of a segment split over several workers, and
// leave segments finished inside one worker (written by the split kernel)
// alone. Used while the grid is at most two waves of resident CTAs.
template <typename QT, int D, int G>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const CombineParams c) {
    __shared__ float s_m[kCombineThreads], s_den[kCombineThreads];
    __shared__ float4 s_num[kCombineThreads];
    griddep_wait();                 // partials come from the split grid
    const int seg = blockIdx.x;
    const int b = seg / c.hkv, kvh = seg - b * c.hkv;
    const int* P = c.ws_prefix;
    const int nb = P[b + 1] - P[b];
    if (nb == 0) {
        zero_segment<QT, D, G>(c, b, kvh);
        return;
    }
    const long long U = (long long)P[c.batch] * c.hkv;
    const long long W = eff_workers(U, c.workers);
    const long long uf = (long long)c.hkv * P[b] + (long long)kvh * nb;
    // workers are below 2^31 (the host caps them)
    const int wf = int(worker_of(uf, U, W)), wl = int(worker_of(uf + nb - 1, U, W));
    if (wf == wl) return;
    merge_segment<QT, D, G>(c, seg, b, kvh, wf, wl, s_m, s_den, s_num);
    // Only now may the next grid start launching: a decode split launched
    // early here would take SM resources while this grid still runs, which
    // measured ~30 % slower steps.
    griddep_launch_dependents();
}

// Large batches: each CTA looks after a run of segs_per_cta consecutive
// segments, so that the grid stays about two waves deep however many
// segments there are (per-CTA overhead, not merging, is what grows with the
// batch). Every warp checks the run 32 segments at a time, one per lane; the
// ballot of the lanes' answers gives all warps the same list of segments to
// zero or merge, so the CTA needs no shared list and no barrier to agree on
// it. Split segments number at most one per worker boundary.
template <typename QT, int D, int G>
__global__ void __launch_bounds__(kCombineThreads, kCombineCtasPerSm)
decode_combine_runs_kernel(const CombineParams c) {
    __shared__ float s_m[kCombineThreads], s_den[kCombineThreads];
    __shared__ float4 s_num[kCombineThreads];
    griddep_wait();                 // partials come from the split grid
    const int* P = c.ws_prefix;
    const long long U = (long long)P[c.batch] * c.hkv;
    const long long W = eff_workers(U, c.workers);
    const int lane = threadIdx.x & 31;
    const int S = c.batch * c.hkv;                     // < 2^31: checked on the host
    const int seg0 = int(blockIdx.x) * c.segs_per_cta;
    for (int base = 0; base < c.segs_per_cta; base += 32) {
        bool split = false, empty = false;
        if (base + lane < c.segs_per_cta && seg0 + base + lane < S) {
            const int seg = seg0 + base + lane;
            const int b = seg / c.hkv, kvh = seg - b * c.hkv;
            const int nb = P[b + 1] - P[b];
            const long long uf = (long long)c.hkv * P[b] + (long long)kvh * nb;
            empty = nb == 0;
            split = !empty && worker_of(uf, U, W) != worker_of(uf + nb - 1, U, W);
        }
        const unsigned empties = __ballot_sync(0xffffffffu, empty);
        for (unsigned todo = __ballot_sync(0xffffffffu, split) | empties; todo; todo &= todo - 1) {
            const int j = __ffs(todo) - 1;
            const int seg = seg0 + base + j;
            const int b = seg / c.hkv, kvh = seg - b * c.hkv;
            if ((empties >> j) & 1u) {
                zero_segment<QT, D, G>(c, b, kvh);
                continue;
            }
            const int nb = P[b + 1] - P[b];
            const long long uf = (long long)c.hkv * P[b] + (long long)kvh * nb;
            merge_segment<QT, D, G>(c, seg, b, kvh, int(worker_of(uf, U, W)),
                                    int(worker_of(uf + nb - 1, U, W)), s_m, s_den, s_num);
            __syncthreads();   // the next segment reuses s_m / s_den / s_num
        }
    }
    griddep_launch_dependents();
}

// ------------------------------------------------------------------- host ---
struct Ops {
    int warp_bytes;
    int warps;             // worker warps per CTA
    int max_ctas_per_sm;   // cap on the default worker count (0 = occupancy)
    cudaError_t (*prepare)(size_t smem);                        // smem attribute
    cudaError_t (*occupancy)(int* blocks, size_t smem);
    void (*split)(const DecodeParams&, int grid, size_t smem, cudaStream_t);
    void (*combine)(const CombineParams&, int grid, cudaStream_t);
};

template <typename KV, typename QT, int D, int G>
struct Impl {
    static cudaError_t prepare(size_t smem) {
        return cudaFuncSetAttribute(decode_split_kernel<KV, QT, D, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    }
    static cudaError_t occupancy(int* blocks, size_t smem) {
        cudaError_t e = prepare(smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks, decode_split_kernel<KV, QT, D, G>, Cfg<KV, D, G>::THREADS, smem);
    }
    static void split(const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
        launch_pdl(decode_split_kernel<KV, QT, D, G>, dim3(grid), dim3(Cfg<KV, D, G>::THREADS),
                   smem, st, p);
    }
    static void combine(const CombineParams& c, int grid, cudaStream_t st) {
        if (c.segs_per_cta == 1)
            launch_pdl(decode_combine_kernel<QT, D, G>, dim3(grid), dim3(kCombineThreads), 0, st, c);
        else
            launch_pdl(decode_combine_runs_kernel<QT, D, G>, dim3(grid), dim3(kCombineThreads), 0,
                       st, c);
    }
    // 16-bit caches at D = 128 default to 2 CTAs (8 worker warps) per SM
    // although 3 fit: on the GQA-8B workload the split kernel read 6.74 TB/s
    // with 8 warps per SM against 6.38 TB/s with 12 (same GPU, back to back),
    // and g = 8, whose shared memory allows only 2, read 6.71 TB/s. INT8
    // (two-block units, 6-warp CTAs) keeps full occupancy: 12 warps per SM
    // read 6.07 TB/s on the INT8 GQA-8B workload, 8 warps 4.2 TB/s.
    static constexpr int kCap = (Elem<KV>::bytes == 2 && D == 128) ? 2 : 0;
    static Ops ops() {
        return Ops{Cfg<KV, D, G>::WARP_BYTES, Cfg<KV, D, G>::WARPS, kCap, prepare, occupancy,
                   split, combine};
    }
};

template <typename KV, typename QT, int D>
bool pick_g(int G, Ops* o) {
    switch (G) {
        case 1: *o = Impl<KV, QT, D, 1>::ops(); return true;
        case 2: *o = Impl<KV, QT, D, 2>::ops(); return true;
        case 4: *o = Impl<KV, QT, D, 4>::ops(); return true;
        case 8: *o = Impl<KV, QT, D, 8>::ops(); return true;
    }
    return false;
}

template <typename KV, typename QT>
bool pick_d(int D, int G, Ops* o) {
    if (D == 128) return pick_g<KV, QT, 128>(G, o);
    if (D == 64) return pick_g<KV, QT, 64>(G, o);
    return false;
}

bool pick_ops(pkv_dtype kv, pkv_dtype q, int D, int G, Ops* o) {
    if (kv == PKV_BF16 && q == PKV_BF16) return pick_d<BF16, BF16>(D, G, o);
    if (kv == PKV_F16 && q == PKV_F16) return pick_d<F16, F16>(D, G, o);
    if (kv == PKV_I8 && q == PKV_BF16) return pick_d<I8, BF16>(D, G, o);
    if (kv == PKV_I8 && q == PKV_F16) return pick_d<I8, F16>(D, G, o);
    return false;
}

struct Layout {
    size_t prefix_off, ml_off, o_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout layout(int batch, int hkv, int G, int D, long long workers) {
    const long long slots = (long long)batch * hkv + workers;
    Layout l;
    l.prefix_off = 0;
    l.ml_off = align256(sizeof(int32_t) * size_t(batch + 1));
    l.o_off = l.ml_off + align256(size_t(slots) * G * 2 * sizeof(float));
    l.total = l.o_off + align256(size_t(slots) * G * D * sizeof(float));
    return l;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks shared by every decode entry point; fills ops and the group size.
pkv_status check_decode(const pkv_cache_desc* c, int batch, int hq, pkv_dtype q_dtype, Ops* ops,
                        int* G) {
    if (!c) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return PKV_ERR_INVALID_ARG;
    if (c->kv_dtype != PKV_F16 && c->kv_dtype != PKV_BF16 && c->kv_dtype != PKV_I8)
        return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (batch < 0 || hq <= 0 || hq % c->num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize || batch > kMaxBatch || c->num_kv_heads > 0xffff)
        return PKV_ERR_UNSUPPORTED;
    if (c->kv_dtype != PKV_I8 && q_dtype != c->kv_dtype) return PKV_ERR_INVALID_ARG;
    *G = hq / c->num_kv_heads;
    if (!pick_ops(c->kv_dtype, q_dtype, c->head_dim, *G, ops)) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

size_t split_smem(const Ops& o, int batch) {
    return size_t(prefix_bytes(batch)) + size_t(o.warps) * o.warp_bytes;
}

// Default worker warps on the current device for this configuration: the
// resident warps, at most max_ctas_per_sm CTAs per SM.
long long default_workers(const Ops& o, int batch) {
    int dev = 0, sms = 0, blocks = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (o.occupancy(&blocks, split_smem(o, batch)) != cudaSuccess || blocks <= 0) return 0;
    if (o.max_ctas_per_sm > 0 && blocks > o.max_ctas_per_sm) blocks = o.max_ctas_per_sm;
    return (long long)sms * blocks * o.warps;
}

pkv_status run_decode(bool do_split, bool do_combine, const void* q, pkv_dtype q_dtype,
                      const void* k_cache, const void* v_cache, const float* k_scales,
                      const float* v_scales, const pkv_cache_desc* cache,
                      const int32_t* block_tables, int32_t mb, const int32_t* context_lens,
                      int32_t batch, int32_t hq, float softmax_scale, void* out, void* workspace,
                      size_t workspace_bytes, int32_t num_parts, uint32_t* dev_status,
                      cudaStream_t stream, const void* k_new = nullptr,
                      const void* v_new = nullptr, uint64_t wait_ns = kWaitLimitNs,
                      int stall_worker = -1, bool check_only = false) {
    Ops ops;
    int G = 0;
    pkv_status s = check_decode(cache, batch, hq, q_dtype, &ops, &G);
    if (s != PKV_OK) return s;
    if (batch == 0) return PKV_OK;
    if (num_parts < 0) return PKV_ERR_INVALID_ARG;
    if (!out || !is_aligned(out, 16)) return PKV_ERR_INVALID_ARG;
    if (do_split || check_only) {
        if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
        if (!is_aligned(q, 16) || !is_aligned(k_cache, 16) || !is_aligned(v_cache, 16) ||
            !is_aligned(block_tables, 4) || !is_aligned(context_lens, 4))
            return PKV_ERR_INVALID_ARG;
        if (cache->kv_dtype == PKV_I8 && (!k_scales || !v_scales || !is_aligned(k_scales, 4) ||
                                          !is_aligned(v_scales, 4)))
            return PKV_ERR_INVALID_ARG;
        if (mb <= 0 || !(softmax_scale == softmax_scale) || softmax_scale > 3.0e38f ||
            softmax_scale < -3.0e38f)
            return PKV_ERR_INVALID_ARG;
        if (dev_status && !is_aligned(dev_status, 4)) return PKV_ERR_INVALID_ARG;
    }
    const long long workers = num_parts > 0 ? num_parts : default_workers(ops, batch);
    if (workers <= 0) return PKV_ERR_CUDA;
    const int D = cache->head_dim, hkv = cache->num_kv_heads;
    const Layout l = layout(batch, hkv, G, D, workers);
    if (!workspace || workspace_bytes < l.total || !is_aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    if (check_only) return PKV_OK;
    char* ws = static_cast<char*>(workspace);
    if (do_split) {
        const size_t smem = split_smem(ops, batch);
        if (ops.prepare(smem) != cudaSuccess) return PKV_ERR_CUDA;
        DecodeParams p;
        p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
        p.k_scales = k_scales; p.v_scales = v_scales;
        p.block_tables = block_tables; p.context_lens = context_lens; p.out = out;
        p.part_o = reinterpret_cast<float*>(ws + l.o_off);
        p.part_ml = reinterpret_cast<float*>(ws + l.ml_off);
        p.ws_prefix = reinterpret_cast<int32_t*>(ws + l.prefix_off);
        p.status = dev_status;
        p.k_new = k_new;
        p.v_new = v_new;
        p.batch = batch; p.hq = hq; p.hkv = hkv; p.mb = mb; p.num_blocks = cache->num_blocks;
        p.workers = int(workers);
        p.qscale = softmax_scale * kLog2e;
        p.wait_ns = wait_ns;
        p.stall_worker = stall_worker;
        const int grid = int((workers + ops.warps - 1) / ops.warps);
        ops.split(p, grid, smem, stream);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (do_combine) {
        CombineParams c;
        c.part_o = reinterpret_cast<const float*>(ws + l.o_off);
        c.part_ml = reinterpret_cast<const float*>(ws + l.ml_off);
        c.ws_prefix = reinterpret_cast<const int32_t*>(ws + l.prefix_off);
        c.out = out;
        c.batch = batch; c.hq = hq; c.hkv = hkv; c.workers = int(workers);
        // One segment per CTA up to two waves of resident combine CTAs
        // (152 SMs x 8); beyond that, runs of segments keep the grid at about
        // two waves.
        const long long segs = (long long)batch * hkv;
        long long spc = (segs + 2431) / 2432;
        spc = spc < 1 ? 1 : (spc > kCombineThreads ? kCombineThreads : spc);
        c.segs_per_cta = int(spc);
        ops.combine(c, int((segs + spc - 1) / spc), stream);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int32_t pkv_decode_default_parts(int32_t device, int32_t batch, int32_t num_q_heads,
                                            const pkv_cache_desc* cache) {
    Ops ops;
    int G = 0;
    const pkv_dtype qd = (cache && cache->kv_dtype == PKV_F16) ? PKV_F16 : PKV_BF16;
    if (check_decode(cache, batch, num_q_heads, qd, &ops, &G) != PKV_OK) return 0;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return 0;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return 0;
    const long long w = default_workers(ops, batch < 1 ? 1 : batch);
    if (prev != device) cudaSetDevice(prev);
    return int32_t(w);
}

extern "C" size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                            const pkv_cache_desc* cache, int32_t num_parts) {
    Ops ops;
    int G = 0;
    const pkv_dtype qd = (cache && cache->kv_dtype == PKV_F16) ? PKV_F16 : PKV_BF16;
    if (check_decode(cache, batch, num_q_heads, qd, &ops, &G) != PKV_OK || num_parts < 0) return 0;
    const long long workers = num_parts > 0 ? num_parts : default_workers(ops, batch < 1 ? 1 : batch);
    if (workers <= 0) return 0;
    return layout(batch, cache->num_kv_heads, G, cache->head_dim, workers).total;
}

extern "C" pkv_status pkv_decode_attn(const void* q, pkv_dtype q_dtype, const void* k_cache,
                                      const void* v_cache, const float* k_scales,
                                      const float* v_scales, const pkv_cache_desc* cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t batch,
                                      int32_t num_q_heads, float softmax_scale, void* out,
                                      void* workspace, size_t workspace_bytes, int32_t num_parts,
                                      uint32_t* dev_status, cudaStream_t stream) {
    return run_decode(true, true, q, q_dtype, k_cache, v_cache, k_scales, v_scales, cache,
                      block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                      softmax_scale, out, workspace, workspace_bytes, num_parts, dev_status, stream);
}

extern "C" pkv_status pkv_decode_split(const void* q, pkv_dtype q_dtype, const void* k_cache,
                                       const void* v_cache, const float* k_scales,
                                       const float* v_scales, const pkv_cache_desc* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t batch,
                                       int32_t num_q_heads, float softmax_scale, void* out,
                                       void* workspace, size_t workspace_bytes, int32_t num_parts,
                                       uint32_t* dev_status, cudaStream_t stream) {
    return run_decode(true, false, q, q_dtype, k_cache, v_cache, k_scales, v_scales, cache,
                      block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                      softmax_scale, out, workspace, workspace_bytes, num_parts, dev_status, stream);
}

namespace pkv {
cudaError_t launch_i8_step_append(const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                  void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                  const int32_t* block_tables, int mb, const int32_t* context_lens,
                                  int batch, int hkv, int D, int num_blocks, uint32_t* status,
                                  cudaStream_t stream);
}

extern "C" pkv_status pkv_decode_step(const void* q, pkv_dtype q_dtype, const void* k_new,
                                      const void* v_new, void* k_cache, void* v_cache,
                                      float* k_scales, float* v_scales,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      int32_t batch, int32_t num_q_heads, float softmax_scale,
                                      void* out, void* workspace, size_t workspace_bytes,
                                      int32_t num_parts, int32_t run_combine,
                                      uint32_t* dev_status, cudaStream_t stream) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    if (run_combine != 0 && run_combine != 1) return PKV_ERR_INVALID_ARG;
    if (batch > 0 && (!k_new || !v_new || !is_aligned(k_new, 16) || !is_aligned(v_new, 16)))
        return PKV_ERR_INVALID_ARG;
    if (cache->kv_dtype != PKV_I8)
        return run_decode(true, run_combine == 1, q, q_dtype, k_cache, v_cache, nullptr, nullptr,
                          cache, block_tables, max_blocks_per_seq, context_lens, batch,
                          num_q_heads, softmax_scale, out, workspace, workspace_bytes, num_parts,
                          dev_status, stream, k_new, v_new);
    // INT8: the step's append kernel (one row per tile), then split [+ combine];
    // every argument is checked (a call that launches nothing) before the append
    pkv_status s = run_decode(true, run_combine == 1, q, q_dtype, k_cache, v_cache, k_scales,
                              v_scales, cache, block_tables, max_blocks_per_seq, context_lens, batch,
                              num_q_heads, softmax_scale, out, workspace, workspace_bytes, num_parts,
                              dev_status, stream, nullptr, nullptr, kWaitLimitNs, -1, true);
    if (s != PKV_OK || batch == 0) return s;
    if (launch_i8_step_append(k_new, v_new, q_dtype, k_cache, v_cache, k_scales, v_scales,
                              block_tables, max_blocks_per_seq, context_lens, batch,
                              cache->num_kv_heads, cache->head_dim, cache->num_blocks, dev_status,
                              stream) != cudaSuccess)
        return PKV_ERR_CUDA;
    return run_decode(true, run_combine == 1, q, q_dtype, k_cache, v_cache, k_scales, v_scales,
                      cache, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                      softmax_scale, out, workspace, workspace_bytes, num_parts, dev_status, stream);
}

extern "C" pkv_status pkv_decode_combine(const pkv_cache_desc* cache, int32_t batch,
                                         int32_t num_q_heads, pkv_dtype out_dtype, void* out,
                                         const void* workspace, size_t workspace_bytes,
                                         int32_t num_parts, cudaStream_t stream) {
    return run_decode(false, true, nullptr, out_dtype, nullptr, nullptr, nullptr, nullptr, cache,
                      nullptr, 0, nullptr, batch, num_q_heads, 1.0f, out,
                      const_cast<void*>(workspace), workspace_bytes, num_parts, nullptr, stream);
}

// ------------------------------------------------ no-allocation variant ---
// pkv_decode_attn_noalloc: the same split + combine, with the scratch taken
// from a fixed array compiled into this file instead of a caller workspace.
#include <cuda.h>

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxContexts = 64;

// Device-resident scratch. In host code this name is only a stand-in; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's address belongs to a CUDA context (each context that loads the
// module has its own copy), so it is cached per (device, context).
struct NoAllocEntry {
    int device;
    CUcontext ctx;
    void* ptr;
};
std::mutex g_noalloc_mu;
NoAllocEntry g_noalloc[kNoAllocMaxContexts];
int g_noalloc_n = 0;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

// Once per (device, context), with that device and context current: resolve
// the array's address. Later calls in the same context reuse it.
pkv_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get) return PKV_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; ctx != nullptr && i < g_noalloc_n; ++i)
        if (g_noalloc[i].device == dev && g_noalloc[i].ctx == ctx) {
            *out = g_noalloc[i].ptr;
            return PKV_OK;
        }
    if (g_noalloc_n == kNoAllocMaxContexts) return PKV_ERR_UNSUPPORTED;
    // Resolving the address also makes the device's primary context current
    // if no context was yet, so the context is read again afterwards.
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PKV_ERR_CUDA;
    g_noalloc[g_noalloc_n++] = NoAllocEntry{dev, ctx, p};
    *out = p;
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attn_noalloc(const void* q, pkv_dtype q_dtype,
                                              const void* k_cache, const void* v_cache,
                                              const float* k_scales, const float* v_scales,
                                              const pkv_cache_desc* cache,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t batch,
                                              int32_t num_q_heads, float softmax_scale,
                                              void* out, int32_t num_parts,
                                              uint32_t* dev_status, cudaStream_t stream) {
    Ops ops;
    int G = 0;
    pkv_status s = check_decode(cache, batch, num_q_heads, q_dtype, &ops, &G);
    if (s != PKV_OK) return s;
    if (batch == 0) return PKV_OK;
    if (num_parts < 0) return PKV_ERR_INVALID_ARG;
    const long long workers = num_parts > 0 ? num_parts : default_workers(ops, batch);
    if (workers <= 0 || workers > 0x7fffffffLL) return workers <= 0 ? PKV_ERR_CUDA : PKV_ERR_INVALID_ARG;
    if (layout(batch, cache->num_kv_heads, G, cache->head_dim, workers).total > kNoAllocScratchBytes)
        return PKV_ERR_WORKSPACE;  // needs more scratch than the built-in array holds
    void* ws = nullptr;
    s = noalloc_scratch(&ws);
    if (s != PKV_OK) return s;
    return run_decode(true, true, q, q_dtype, k_cache, v_cache, k_scales, v_scales, cache,
                      block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                      softmax_scale, out, ws, kNoAllocScratchBytes, int32_t(workers), dev_status,
                      stream);
}

// ------------------------------------------------------------- test hook ---
#include "../../include/pkv_testing.h"

extern "C" pkv_status pkv_testing_decode_attn_stall(
    const void* q, pkv_dtype q_dtype, const void* k_cache, const void* v_cache,
    const float* k_scales, const float* v_scales, const pkv_cache_desc* cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t batch, int32_t num_q_heads, float softmax_scale, void* out, void* workspace,
    size_t workspace_bytes, int32_t num_parts, uint64_t wait_limit_ns, int32_t stall_worker,
    uint32_t* dev_status, cudaStream_t stream) {
    if (wait_limit_ns > kWaitLimitNs || stall_worker < -1) return PKV_ERR_INVALID_ARG;
    return run_decode(true, true, q, q_dtype, k_cache, v_cache, k_scales, v_scales, cache,
                      block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                      softmax_scale, out, workspace, workspace_bytes, num_parts, dev_status,
                      stream, nullptr, nullptr, wait_limit_ns, stall_worker);
}
