// Multi-query paged attention: n_b new query tokens per sequence, causal
// among themselves, over the paged KV cache (which already holds them).
//
// The target model of speculative decoding scores the draft's K tokens plus
// one in a single batched pass (Continuous-Batching-LLM-Inference-Engine
// README, feature list "Speculative decoding"); a continuous-batching
// scheduler mixes decode tokens with prefill chunks (mini-inference-engine
// overview, "decode tokens and prefill chunks"). Query i of sequence b sits at
// position L_b - n_b + i and attends to positions 0 .. L_b - n_b + i.
//
// GB300 design. With n_b queries the g query heads of a KV head form
// n_b * g rows that share every K/V tile: a real dense contraction, so the
// math runs on the tensor cores (mma.sync m16n8k16, bf16/fp16 in, fp32
// accumulate), FlashAttention-2 style:
// * a CTA = NW consumer warps (16 rows each; a row tile of RT = 16 NW rows)
//   + 1 producer warp. Work units are (sequence, kv head, row tile, block)
//   with the blocks the tile's rows can see; the unit stream is cut into
//   equal ranges per CTA (as in the decode kernel).
// * The producer issues 2-D TMA tensor copies (cp.async.bulk.tensor) of each
//   16-token K and V tile in 64-column boxes with the 128-byte swizzle into a
//   ring of stages (full/empty mbarriers); consumers read B fragments with
//   ldmatrix (K) and ldmatrix.trans (V) without bank conflicts.
// * S = Q K^T (Q A fragments in registers), causal/length mask, online
//   softmax in base 2 per row, P re-packed in registers as the A operand of
//   O += P V. Rows of a piece that crosses ranges leave (m, l, o) partials;
//   a combine kernel merges them.
//
// This header holds the mma.sync split kernel and its combine; mq.cu
// instantiates them for fp16 / bf16 caches (and holds the tcgen05 kernel for
// long query runs), mq_i8.cu for INT8 caches, in parallel compilations. The
// short-run kernels (query rows on the MMA's N side) live in mq_t.cu and use
// the partition, prefix and combine defined here.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace pkv {

// The split kernel's parameters. Kept at 128 bytes: grown to 160 bytes with
// fields the 16-bit kernels never read, the same 16-bit split kernel ran 8 %
// slower on the speculative-verification workload (same registers, same
// code; measured back to back on one GPU).
struct MqParams {
    const void* q;               // [total_q, hq, D]
    const int32_t* cu_q;         // [B + 1]
    const int32_t* block_tables; // [B, mb]
    const int32_t* context_lens; // [B]
    void* out;                   // [total_q, hq, D]
    float* part_o;               // [slots, RT, D]
    float* part_ml;              // [slots, RT, 2]
    int32_t* ws_prefix;          // [B + 1] units before each sequence
    uint32_t* status;
    int batch, hq, hkv, mb, num_blocks, workers, tmax, max_q;
    float qscale;                // softmax_scale * log2(e)
    uint64_t wait_ns;            // limit of each bounded wait
    int stall_cta;               // test hook: this CTA's first unit (split kernel) or
                                 // first chunk (tcgen05 kernel) expects 16 bytes no
                                 // copy delivers, so its wait runs out (-1: none)
};
static_assert(sizeof(MqParams) <= 128, "keep the split kernel's parameters small");

// Where a split kernel reads K and V tiles: 16-bit caches through 2-D tensor
// maps (TMA, 128-byte swizzle), INT8 caches as plain pointers (1-D bulk
// copies of whole tiles) with their per-(block, kv head) scales.
struct MqI8Src {
    const void* cache;
    const float* scales;
};
// An INT8 cache read through a 2-D tensor map (128-byte rows of codes, the
// 128-byte swizzle), with its scales: the short-run INT8 kernel's source.
struct MqI8Map {
    CUtensorMap map;
    const float* scales;
};

struct MqCombine {
    const float* part_o;
    const float* part_ml;
    const int32_t* ws_prefix;
    const int32_t* cu_q;
    const int32_t* context_lens;
    void* out;
    int batch, hq, hkv, mb, workers, tmax, max_q;
};

struct MqOps {
    int fixed_smem, rt, threads;
    cudaError_t (*prepare)(size_t smem);
    cudaError_t (*occupancy)(int* blocks, size_t smem);
    // k_src, v_src: as `src` says; the int is the number of CTAs
    cudaError_t (*split)(const void* k_src, const void* v_src, const MqParams&, int, size_t,
                         cudaStream_t);
    cudaError_t (*combine)(const MqCombine&, int, cudaStream_t);
    int wpc;               // workers per CTA
    int src;               // kMqSrc*: how the split kernel reads K and V
};
constexpr int kMqSrcMap = 0;     // CUtensorMap of a 16-bit cache
constexpr int kMqSrcRaw = 1;     // MqI8Src: plain pointers (INT8 caches)
constexpr int kMqSrcI8Map = 2;   // MqI8Map: tensor map of an INT8 cache + its scales

// The INT8 split kernels (mq_i8.cu): ops of the variant for this q dtype,
// head dim, group size and tile height; false if not built.
bool mq_pick_i8(pkv_dtype q_dtype, int D, int G, int nw, MqOps* o);
// The short-run split kernels (mq_t.cu): query rows on the MMA's N side in nt
// tiles of 8 (at most 24 rows), for fp16 / bf16 caches (q of the cache type)
// and for INT8 caches at head_dim 128 (q bf16 or fp16); false if not built.
bool mqt_pick(pkv_dtype kv_dtype, pkv_dtype q_dtype, int D, int G, int nt, MqOps* o);

namespace {


constexpr uint64_t kMqWaitNs = 4000000000ull;
constexpr int kMqMaxBatch = 4096;
constexpr float kMqLog2e = 1.4426950408889634f;


// Blocks the rows of row tile t can see: its last query sits at position
// L - n + min(n - 1, ((t + 1) RT - 1) / G).
__host__ __device__ __forceinline__ int tile_blocks(int n, int L, int t, int RT, int G) {
    const int q_last = min(n - 1, ((t + 1) * RT - 1) / G);
    return (L - n + q_last) / kBlockSize + 1;
}

// Queries and length of sequence b, checked: max_q >= n >= 0, L >= n and L
// within the table; an inconsistent sequence is treated as empty (flagged).
__device__ __forceinline__ void seq_shape_raw(const int32_t* cu_q, const int32_t* lens, int b,
                                              int mb, int max_q, int& n, int& L, bool& bad) {
    n = cu_q[b + 1] - cu_q[b];
    L = lens[b];
    bad = n < 0 || n > max_q || L < n || L > mb * kBlockSize;
    if (bad) n = L = 0;
}
__device__ __forceinline__ void seq_shape(const MqParams& p, int b, int& n, int& L, bool flag) {
    bool bad;
    seq_shape_raw(p.cu_q, p.context_lens, b, p.mb, p.max_q, n, L, bad);
    if (bad && flag) flag_status(p.status, PKV_DEV_BAD_LENGTH);
}

// Units of one kv head of sequence b: sum over its row tiles of tile_blocks.
__device__ __forceinline__ int seq_units_per_head(int n, int L, int RT, int G) {
    if (n == 0) return 0;
    const int T = (n * G + RT - 1) / RT;
    int s = 0;
    for (int t = 0; t < T; ++t) s += tile_blocks(n, L, t, RT, G);
    return s;
}

// prefix[b] = units (all kv heads) before sequence b; all threads of the CTA.
template <int NT>
__device__ void mq_build_prefix(const MqParams& p, int* warp_tot, int* prefix, int RT, int G) {
    const int t = threadIdx.x;
    const int chunk = (p.batch + NT - 1) / NT;
    const int lo = min(p.batch, t * chunk), hi = min(p.batch, lo + chunk);
    const bool flag = blockIdx.x == 0;
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
        int n, L;
        seq_shape(p, i, n, L, flag);
        sum += p.hkv * seq_units_per_head(n, L, RT, G);
    }
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
    for (int i = lo; i < hi; ++i) {
        prefix[i] = run;
        int n, L;
        seq_shape(p, i, n, L, false);
        run += p.hkv * seq_units_per_head(n, L, RT, G);
    }
    if (t == NT - 1) prefix[p.batch] = run;
    __syncthreads();
    if (blockIdx.x == 0)
        for (int i = t; i <= p.batch; i += NT) p.ws_prefix[i] = prefix[i];
}

// Unit u -> (b, kv head, row tile t, block j, n, L).
__device__ __forceinline__ void mq_decode_unit(const MqParams& p, const int* prefix, int u, int RT,
                                               int G, int& b, int& kvh, int& t, int& j, int& n,
                                               int& L) {
    int lo = 0;
    for (int step = 1 << 12; step; step >>= 1)  // kMqMaxBatch = 2^12
        if (lo + step < p.batch && prefix[lo + step] <= u) lo += step;
    b = lo;
    seq_shape(p, b, n, L, false);
    const int per_head = seq_units_per_head(n, L, RT, G);
    int r = u - prefix[b];
    kvh = r / per_head;
    r -= kvh * per_head;
    t = 0;
    for (;;) {
        const int nb = tile_blocks(n, L, t, RT, G);
        if (r < nb) break;
        r -= nb;
        ++t;
    }
    j = r;
}

// ------------------------------------------------------------ PTX helpers ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Byte offset of (row r, 16-byte chunk c) inside one 16 x 128-byte sub-tile
// written by TMA with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int D, int NW, int ES>
struct MqCfg {
    // ring depth (6 stages measured slower than 4 for the 32-row variant)
    static constexpr int NS = 4;
    static constexpr int RT = 16 * NW;                 // rows per tile
    static constexpr int NT = 32 * (NW + 1);           // threads: NW consumers + producer
    static constexpr int SUB = 16 * 128;               // one 16 x 64-element sub-tile (16-bit)
    static constexpr int NSUB = D / 64;                // sub-tiles per K (or V) tile
    // 16-bit caches: NSUB swizzled 2-D boxes; INT8: the tile's 16 rows of D
    // codes as they lie in the cache (one 1-D bulk copy)
    static constexpr int TILE = ES == 2 ? NSUB * SUB : kBlockSize * D;
    static constexpr int STAGE = 2 * TILE;             // K then V
    static constexpr int OFF_FULL = NS * STAGE;
    static constexpr int OFF_EMPTY = OFF_FULL + NS * 8;
    static constexpr int OFF_META = OFF_EMPTY + NS * 8;   // 2 x int4 per stage
    static constexpr int OFF_SCL = OFF_META + NS * 32;    // INT8: the block's K, V scales
    static constexpr int OFF_SCAN = OFF_SCL + NS * 8;
    static constexpr int OFF_PREFIX = OFF_SCAN + 32;
    // dynamic shared memory: alignment slack + the layout above + the prefix
    static constexpr int fixed_bytes() { return 1024 + OFF_PREFIX; }
    static_assert(D == 64 || D == 128, "head_dim");
};

__device__ __forceinline__ long long mq_eff_workers(long long U, long long W) {
    const long long cap = U / 4;   // at least 4 units per range: ranges are never empty
    return cap < 1 ? 1 : (cap < W ? cap : W);
}

template <typename KV>
using MqSrc = typename std::conditional<Elem<KV>::bytes == 1, MqI8Src, CUtensorMap>::type;

template <typename KV, typename QT, int D, int G, int NW>
__global__ void __launch_bounds__(32 * (NW + 1))
mq_split_kernel(const __grid_constant__ MqSrc<KV> tmk, const __grid_constant__ MqSrc<KV> tmv,
                const MqParams p) {
    constexpr bool kI8 = Elem<KV>::bytes == 1;
    using C = MqCfg<D, NW, Elem<KV>::bytes>;
    constexpr int NS = C::NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
    int4* meta = reinterpret_cast<int4*>(smem + C::OFF_META);
    float2* scl = reinterpret_cast<float2*>(smem + C::OFF_SCL);
    int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_addr(&full[s]), kI8 ? 2 : 1);   // INT8: + the scales' cp.async
            mbar_init(smem_addr(&empty[s]), NW);
        }
        fence_mbar_init();
    }
    mq_build_prefix<C::NT>(p, reinterpret_cast<int*>(smem + C::OFF_SCAN), prefix, C::RT, G);
    const long long U = prefix[p.batch];
    const long long W = mq_eff_workers(U, p.workers);
    const long long wk = blockIdx.x;
    if (wk >= W || U == 0) return;
    const int u0 = int(wk * U / W), u1 = int((wk + 1) * U / W);

    if (warp == NW) {
        // ------------------------------------------------------ producer ---
        auto fetch = [&](int base, int& b, int& kvh, int& t, int& j, int& n, int& L, int& blk,
                         int& cu) {
            const int u = base + lane;
            if (u < u1) {
                mq_decode_unit(p, prefix, u, C::RT, G, b, kvh, t, j, n, L);
                blk = __ldg(p.block_tables + (long long)b * p.mb + j);
                cu = __ldg(p.cu_q + b);
            } else {
                b = kvh = t = j = n = L = cu = 0;
                blk = -1;
            }
        };
        int cbase = u0;
        int cb, ck, ct, cj, cn, cL, cblk, ccu, xb, xk, xt, xj, xn, xL, xblk, xcu;
        fetch(cbase, cb, ck, ct, cj, cn, cL, cblk, ccu);
        fetch(cbase + 32, xb, xk, xt, xj, xn, xL, xblk, xcu);
        uint32_t parity = 0;
        int s = 0;
        for (int u = u0; u < u1; ++u, s = (s + 1 == NS) ? 0 : s + 1) {
            int idx = u - cbase;
            if (idx >= 32) {
                cbase += 32;
                cb = xb; ck = xk; ct = xt; cj = xj; cn = xn; cL = xL; cblk = xblk; ccu = xcu;
                fetch(cbase + 32, xb, xk, xt, xj, xn, xL, xblk, xcu);
                idx -= 32;
            }
            const int b = __shfl_sync(kFull, cb, idx), kvh = __shfl_sync(kFull, ck, idx);
            const int t = __shfl_sync(kFull, ct, idx), j = __shfl_sync(kFull, cj, idx);
            const int n = __shfl_sync(kFull, cn, idx), L = __shfl_sync(kFull, cL, idx);
            const int blk = __shfl_sync(kFull, cblk, idx), cu = __shfl_sync(kFull, ccu, idx);
            if (u - u0 >= NS) {  // wait until every consumer released this stage
                const bool ok = mbar_wait_bounded(smem_addr(&empty[s]), (parity >> s) & 1u, p.wait_ns);
                parity ^= 1u << s;
                if (!__all_sync(kFull, ok)) {   // records where it gave up: bit 9
                    if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT | 0x200u);
                    return;
                }
            }
            if (lane == 0) {
                const uint32_t bar = smem_addr(&full[s]);
                const bool valid = unsigned(blk) < unsigned(p.num_blocks);
                const uint32_t extra = (u == u0 && wk == p.stall_cta) ? 16u : 0u;
                meta[2 * s] = make_int4(b, kvh, t, j);
                // (n, L, cu_q[b], flags: bit 0 = block valid, bit 1 = first unit of a piece)
                meta[2 * s + 1] = make_int4(n, L, cu, (valid ? 1 : 0) | ((u == u0 || j == 0) ? 2 : 0));
                if (valid) {
                    unsigned char* st = smem + s * C::STAGE;
                    mbar_arrive_expect_tx(bar, C::STAGE + extra);
                    if constexpr (kI8) {
                        const long long tile = (long long)blk * p.hkv + kvh;
                        bulk_g2s(smem_addr(st), static_cast<const char*>(tmk.cache) + tile * C::TILE,
                                 C::TILE, bar);
                        bulk_g2s(smem_addr(st + C::TILE),
                                 static_cast<const char*>(tmv.cache) + tile * C::TILE, C::TILE, bar);
                        cp_async_4(smem_addr(&scl[s].x), tmk.scales + tile);
                        cp_async_4(smem_addr(&scl[s].y), tmv.scales + tile);
                        cp_async_arrive_noinc(bar);
                    } else {
                        const int y = (blk * p.hkv + kvh) * kBlockSize;
#pragma unroll
                        for (int sub = 0; sub < C::NSUB; ++sub) {
                            tma_load_2d(smem_addr(st + sub * C::SUB), &tmk, 64 * sub, y, bar);
                            tma_load_2d(smem_addr(st + C::TILE + sub * C::SUB), &tmv, 64 * sub, y,
                                        bar);
                        }
                    }
                } else {
                    flag_status(p.status, PKV_DEV_BAD_BLOCK);
                    if (extra) mbar_arrive_expect_tx(bar, extra);
                    else mbar_arrive(bar);
                    if constexpr (kI8) mbar_arrive(bar);
                }
            }
        }
        return;
    }

    if constexpr (kI8) {
    // ------------------------------------------------- consumers (INT8) ---
    // Codes c enter the MMAs as the exact fp16 value 1152 + c (the byte XOR
    // 0x80 as the low mantissa byte of 1024), as in the decode kernel:
    //  * S = Q K^T with q rounded to fp16 and the contraction index permuted
    //    so that lane tq's 16-byte chunk of a K row (dims 16 tq .. + 16, and
    //    64 + 16 tq .. for D = 128) serves four k-steps; k-step kk of lane tq
    //    takes dims d0 = 16 tq + 4 (kk % 4) + 64 (kk / 4) .. d0 + 3. The
    //    1152 bias adds 1152 sum_d q_d to every score of a row; it comes off
    //    before the block's K scale.
    //  * O += P V with V as the B operand: the output dims are permuted so
    //    that lane gq's B columns are dims gq D/8 .. + D/8 (one chunk of each
    //    of its four token rows, bytes interleaved with prmt), and the
    //    accumulator of n-tile nd, column n holds dim n D/8 + nd. P enters as
    //    one fp16 value w = rn16(P s_v) (s_v the block's V scale), and
    //    1152 sum_t w_t comes off each row when the piece is written.
    //  * Rows past the context need no zeroing: every byte is a finite code
    //    and its P is exactly 0.
    const int gq = lane >> 2, tq = lane & 3;
    constexpr int DL = D / 8;                     // output dims per lane column
    uint32_t qa[D / 16][4];                       // fp16 Q A fragments (permuted k)
    float o[D / 8][4];                            // O accumulators (permuted dims)
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float kb0 = 0.f, kb1 = 0.f;                   // 1152 sum_d q_d of rows gq, gq + 8
    float pw0 = 0.f, pw1 = 0.f;                   // sum_t w_t of the lane's tokens, per row
    int vexp = 0;                                 // O in units of 2^vexp (see decode)
    float vmul = 1.f;
    int pb = -1, pk = 0, pt = 0, pn = 0, pL = 0, first_j = 0, last_j = 0;
    bool v0 = false, v1 = false;
    bool wact = false;
    int pos0 = 0, pos1 = 0;
    long long orow0 = 0, orow1 = 0;

    auto finalize = [&]() {
        float a = l0, c = l1, w0 = pw0, w1 = pw1;
        a += __shfl_xor_sync(kFull, a, 1); a += __shfl_xor_sync(kFull, a, 2);
        c += __shfl_xor_sync(kFull, c, 1); c += __shfl_xor_sync(kFull, c, 2);
        w0 += __shfl_xor_sync(kFull, w0, 1); w0 += __shfl_xor_sync(kFull, w0, 2);
        w1 += __shfl_xor_sync(kFull, w1, 1); w1 += __shfl_xor_sync(kFull, w1, 2);
        if (!v0 && !v1) return;
        const float up = ldexpf(1.f, vexp);
        const float cb0 = 1152.f * w0, cb1 = 1152.f * w1;
        const bool whole = first_j == 0 && last_j == tile_blocks(pn, pL, pt, C::RT, G) - 1;
        // lane (gq, tq) holds dims (2 tq + cc) DL + nd, nd = 0 .. DL - 1, of rows gq
        // (o[nd][cc]) and gq + 8 (o[nd][2 + cc])
        if (whole) {
            const float i0 = a > 0.f ? up / a : 0.f, i1 = c > 0.f ? up / c : 0.f;
            uint32_t* out = static_cast<uint32_t*>(p.out);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int nd = 0; nd < DL; nd += 2) {
                    const int d = (2 * tq + cc) * DL + nd;
                    if (v0) out[(orow0 + d) / 2] = pack2<QT>((o[nd][cc] - cb0) * i0, (o[nd + 1][cc] - cb0) * i0);
                    if (v1) out[(orow1 + d) / 2] = pack2<QT>((o[nd][2 + cc] - cb1) * i1,
                                                             (o[nd + 1][2 + cc] - cb1) * i1);
                }
        } else {
            const long long slot = ((long long)pb * p.hkv + pk) * p.tmax + pt + wk;
            const long long r0 = slot * C::RT + warp * 16 + gq, r1 = r0 + 8;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int nd = 0; nd < DL; nd += 2) {
                    const int d = (2 * tq + cc) * DL + nd;
                    if (v0) *reinterpret_cast<float2*>(p.part_o + r0 * D + d) =
                                make_float2((o[nd][cc] - cb0) * up, (o[nd + 1][cc] - cb0) * up);
                    if (v1) *reinterpret_cast<float2*>(p.part_o + r1 * D + d) =
                                make_float2((o[nd][2 + cc] - cb1) * up, (o[nd + 1][2 + cc] - cb1) * up);
                }
            if (tq == 0) {
                if (v0) *reinterpret_cast<float2*>(p.part_ml + r0 * 2) = make_float2(m0, a);
                if (v1) *reinterpret_cast<float2*>(p.part_ml + r1 * 2) = make_float2(m1, c);
            }
        }
    };

    uint32_t parity = 0;
    int s = 0;
    bool aborted = false;
    for (int u = u0; u < u1; ++u, s = (s + 1 == NS) ? 0 : s + 1) {
        const bool got = mbar_wait_bounded(smem_addr(&full[s]), (parity >> s) & 1u, p.wait_ns);
        parity ^= 1u << s;
        if (!__all_sync(kFull, got)) {          // records where it gave up: bit 8
            if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT | 0x100u);
            aborted = true;
            break;
        }
        const int4 ma = meta[2 * s], mb = meta[2 * s + 1];
        if (mb.w & 2) {  // first unit of a new piece: load the warp's Q rows
            if (pb >= 0) finalize();
            pb = ma.x; pk = ma.y; pt = ma.z; first_j = ma.w; pn = mb.x; pL = mb.y;
            const int rr0 = pt * C::RT + warp * 16 + gq, rr1 = rr0 + 8;
            v0 = rr0 < pn * G;
            v1 = rr1 < pn * G;
            wact = pt * C::RT + warp * 16 < pn * G;   // warp-uniform
            const int cu = mb.z;
            orow0 = ((long long)(cu + rr0 / G) * p.hq + pk * G + rr0 % G) * D;
            orow1 = ((long long)(cu + rr1 / G) * p.hq + pk * G + rr1 % G) * D;
            pos0 = pL - pn + rr0 / G;
            pos1 = pL - pn + rr1 / G;
            const uint4* q16 = static_cast<const uint4*>(p.q);   // 8 values per uint4
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                // dims 64 h + 16 tq .. + 16 of both rows: k-steps 4 h .. 4 h + 3
                uint4 x0[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                uint4 x1[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                if (v0) { x0[0] = __ldg(q16 + (orow0 + 64 * h + 16 * tq) / 8);
                          x0[1] = __ldg(q16 + (orow0 + 64 * h + 16 * tq + 8) / 8); }
                if (v1) { x1[0] = __ldg(q16 + (orow1 + 64 * h + 16 * tq) / 8);
                          x1[1] = __ldg(q16 + (orow1 + 64 * h + 16 * tq + 8) / 8); }
                const uint32_t* w0 = reinterpret_cast<const uint32_t*>(x0);
                const uint32_t* w1 = reinterpret_cast<const uint32_t*>(x1);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {   // k-step 4 h + k4: dims 4 k4 .. + 4 of the chunk
                    uint32_t f[4];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float2 a = unpack2(QT{}, w0[2 * k4 + e]), b = unpack2(QT{}, w1[2 * k4 + e]);
                        f[e] = pack2<F16>(a.x, a.y);
                        f[2 + e] = pack2<F16>(b.x, b.y);
                        const float2 ra = unpack2(F16{}, f[e]), rb = unpack2(F16{}, f[2 + e]);
                        s0 += ra.x + ra.y;
                        s1 += rb.x + rb.y;
                    }
                    uint32_t* qf = qa[4 * h + k4];
                    qf[0] = f[0]; qf[1] = f[2]; qf[2] = f[1]; qf[3] = f[3];
                }
            }
            s0 += __shfl_xor_sync(kFull, s0, 1); s0 += __shfl_xor_sync(kFull, s0, 2);
            s1 += __shfl_xor_sync(kFull, s1, 1); s1 += __shfl_xor_sync(kFull, s1, 2);
            kb0 = 1152.f * s0;
            kb1 = 1152.f * s1;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            pw0 = pw1 = 0.f;
            vexp = 0;
            vmul = 1.f;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        }
        last_j = ma.w;
        if ((mb.w & 1) && wact) {
            const unsigned char* kt = smem + s * C::STAGE;
            const unsigned char* vt = kt + C::TILE;
            const int j = ma.w;
            const float2 sv = scl[s];
            float vsc = sv.y;
            if (vsc * vmul >= 16384.f) {   // warp-uniform; raise vexp, rescale O exactly
                int ex;
                frexpf(vsc, &ex);
                const int nexp = ex - 14;
                const float r = ldexpf(1.f, vexp - nexp);
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][0] *= r; o[nd][1] *= r; o[nd][2] *= r; o[nd][3] *= r;
                }
                pw0 *= r; pw1 *= r;
                vexp = nexp;
                vmul = ldexpf(1.f, -nexp);
            }
            vsc *= vmul;
            // S = Q K^T for tokens gq (n-tile 0) and gq + 8 (n-tile 1)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int nn = 0; nn < 2; ++nn) {
                const unsigned char* row = kt + (gq + 8 * nn) * D + 16 * tq;
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    const uint4 y = *reinterpret_cast<const uint4*>(row + 64 * h);
                    const uint32_t w[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const uint32_t u4 = w[k4] ^ 0x80808080u;
                        const uint32_t* a = qa[4 * h + k4];
                        mma_16816_f16(sc[nn], a[0], a[1], a[2], a[3], i8x2_biased_h2(u4, 0x4140),
                                      i8x2_biased_h2(u4, 0x4342));
                    }
                }
            }
            // the lane's four V rows: tokens 2tq, 2tq + 1, 2tq + 8, 2tq + 9, dims gq DL ..
            uint32_t vw[4][DL / 4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const unsigned char* row = vt + (2 * tq + (i & 1) + 8 * (i >> 1)) * D + gq * DL;
                if constexpr (DL == 16) {
                    const uint4 x = *reinterpret_cast<const uint4*>(row);
                    vw[i][0] = x.x; vw[i][1] = x.y; vw[i][2] = x.z; vw[i][3] = x.w;
                } else {
                    const uint2 x = *reinterpret_cast<const uint2*>(row);
                    vw[i][0] = x.x; vw[i][1] = x.y;
                }
            }
            // causal + length mask, online softmax per row (base 2)
            const float sk = p.qscale * sv.x;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = kBlockSize * j + 8 * nn + 2 * tq + e;
                    sc[nn][e] = (v0 && col <= pos0) ? (sc[nn][e] - kb0) * sk : -INFINITY;
                    sc[nn][2 + e] = (v1 && col <= pos1) ? (sc[nn][2 + e] - kb1) * sk : -INFINITY;
                    mx0 = fmaxf(mx0, sc[nn][e]);
                    mx1 = fmaxf(mx1, sc[nn][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
            const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
            m0 = n0;
            m1 = n1;
            float pr[2][4];
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mr = e < 2 ? n0 : n1;
                    pr[nn][e] = (sc[nn][e] == -INFINITY) ? 0.f : fast_exp2(sc[nn][e] - mr);
                }
            l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
            l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
            // P A fragments: rows gq (k 2tq, 2tq + 1 | + 8), gq + 8; one fp16 part
            uint32_t pa[4];
            float ws0 = 0.f, ws1 = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                pa[k] = pack2<F16>(pr[k >> 1][2 * (k & 1)] * vsc, pr[k >> 1][2 * (k & 1) + 1] * vsc);
                const float2 r = unpack2(F16{}, pa[k]);
                if (k & 1) ws1 += r.x + r.y;
                else ws0 += r.x + r.y;
            }
            pw0 = fmaf(pw0, a0, ws0);
            pw1 = fmaf(pw1, a1, ws1);
            if (__any_sync(kFull, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][0] *= a0; o[nd][1] *= a0; o[nd][2] *= a1; o[nd][3] *= a1;
                }
            }
            // O += P V: n-tile nd takes dim gq DL + nd of the lane's rows
#pragma unroll
            for (int k = 0; k < DL / 4; ++k)
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {   // bytes 0-1 -> dims 4k, 4k + 1; 2-3 -> 4k + 2, 4k + 3
                    const uint32_t sel = hb ? 0x7362u : 0x5140u;
                    const uint32_t x = __byte_perm(vw[0][k], vw[1][k], sel) ^ 0x80808080u;
                    const uint32_t y = __byte_perm(vw[2][k], vw[3][k], sel) ^ 0x80808080u;
                    const int nd = 4 * k + 2 * hb;
                    mma_16816_f16(o[nd], pa[0], pa[1], pa[2], pa[3], i8x2_biased_h2(x, 0x4140),
                                  i8x2_biased_h2(y, 0x4140));
                    mma_16816_f16(o[nd + 1], pa[0], pa[1], pa[2], pa[3], i8x2_biased_h2(x, 0x4342),
                                  i8x2_biased_h2(y, 0x4342));
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    if (!aborted && pb >= 0) finalize();
    } else {
    // ---------------------------------------------------------- consumers ---
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t qa[D / 16][4];          // Q A fragments of the warp's 16 rows
    float o[D / 8][4];               // O accumulators: rows gq (0,1), gq + 8 (2,3)
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int pb = -1, pk = 0, pt = 0, pn = 0, pL = 0, first_j = 0, last_j = 0;
    bool v0 = false, v1 = false;     // rows gq / gq + 8 exist (per lane)
    bool wact = false;               // the warp covers at least one row (warp-uniform)
    int pos0 = 0, pos1 = 0;          // their query positions
    long long orow0 = 0, orow1 = 0;  // their q / out element offsets

    auto finalize = [&]() {
        float a = l0, c = l1;
        a += __shfl_xor_sync(kFull, a, 1); a += __shfl_xor_sync(kFull, a, 2);
        c += __shfl_xor_sync(kFull, c, 1); c += __shfl_xor_sync(kFull, c, 2);
        if (!v0 && !v1) return;
        const bool whole = first_j == 0 && last_j == tile_blocks(pn, pL, pt, C::RT, G) - 1;
        if (whole) {
            const float i0 = a > 0.f ? 1.f / a : 0.f, i1 = c > 0.f ? 1.f / c : 0.f;
            uint32_t* out = static_cast<uint32_t*>(p.out);
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                if (v0) out[(orow0 + 8 * nd + 2 * tq) / 2] = pack2<KV>(o[nd][0] * i0, o[nd][1] * i0);
                if (v1) out[(orow1 + 8 * nd + 2 * tq) / 2] = pack2<KV>(o[nd][2] * i1, o[nd][3] * i1);
            }
        } else {
            const long long slot = ((long long)pb * p.hkv + pk) * p.tmax + pt + wk;
            const long long r0 = slot * C::RT + warp * 16 + gq, r1 = r0 + 8;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                if (v0) *reinterpret_cast<float2*>(p.part_o + r0 * D + 8 * nd + 2 * tq) =
                            make_float2(o[nd][0], o[nd][1]);
                if (v1) *reinterpret_cast<float2*>(p.part_o + r1 * D + 8 * nd + 2 * tq) =
                            make_float2(o[nd][2], o[nd][3]);
            }
            if (tq == 0) {
                if (v0) *reinterpret_cast<float2*>(p.part_ml + r0 * 2) = make_float2(m0, a);
                if (v1) *reinterpret_cast<float2*>(p.part_ml + r1 * 2) = make_float2(m1, c);
            }
        }
    };

    uint32_t parity = 0;
    int s = 0;
    bool aborted = false;
    for (int u = u0; u < u1; ++u, s = (s + 1 == NS) ? 0 : s + 1) {
        const bool got = mbar_wait_bounded(smem_addr(&full[s]), (parity >> s) & 1u, p.wait_ns);
        parity ^= 1u << s;
        if (!__all_sync(kFull, got)) {          // records where it gave up: bit 8
            if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT | 0x100u);
            aborted = true;
            break;
        }
        const int4 ma = meta[2 * s], mb = meta[2 * s + 1];
        if (mb.w & 2) {  // first unit of a new piece: load the warp's Q rows
            if (pb >= 0) finalize();
            pb = ma.x; pk = ma.y; pt = ma.z; first_j = ma.w; pn = mb.x; pL = mb.y;
            const int rr0 = pt * C::RT + warp * 16 + gq, rr1 = rr0 + 8;
            v0 = rr0 < pn * G;
            v1 = rr1 < pn * G;
            // warp-uniform: the collective ldmatrix / mma / shuffles below
            // must be reached by all 32 lanes or by none
            wact = pt * C::RT + warp * 16 < pn * G;
            const int cu = mb.z;
            orow0 = ((long long)(cu + rr0 / G) * p.hq + pk * G + rr0 % G) * D;
            orow1 = ((long long)(cu + rr1 / G) * p.hq + pk * G + rr1 % G) * D;
            pos0 = pL - pn + rr0 / G;
            pos1 = pL - pn + rr1 / G;
            const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qa[kk][0] = v0 ? __ldg(q32 + (orow0 + 16 * kk + 2 * tq) / 2) : 0u;
                qa[kk][1] = v1 ? __ldg(q32 + (orow1 + 16 * kk + 2 * tq) / 2) : 0u;
                qa[kk][2] = v0 ? __ldg(q32 + (orow0 + 16 * kk + 2 * tq + 8) / 2) : 0u;
                qa[kk][3] = v1 ? __ldg(q32 + (orow1 + 16 * kk + 2 * tq + 8) / 2) : 0u;
            }
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        }
        last_j = ma.w;
        bool zeroed = false;
        if ((mb.w & 1) && wact) {
            unsigned char* kt = smem + s * C::STAGE;
            unsigned char* vt = kt + C::TILE;
            const int j = ma.w;
            const int nvt = min(kBlockSize, pL - kBlockSize * j);   // tokens present in the tile
            if (nvt < kBlockSize) {  // stale rows may hold NaN: P.V must read zeros there
                for (int off = lane * 16; off < (kBlockSize - nvt) * 128; off += 32 * 16)
#pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub)
                        *reinterpret_cast<uint4*>(vt + sub * C::SUB + nvt * 128 + off) =
                            make_uint4(0u, 0u, 0u, 0u);
                zeroed = true;
                __syncwarp();
            }
            // S = Q K^T for the 16 tokens of the tile (two n8 tiles)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int tok = ((mi & 2) ? 8 : 0) + r8, c = 2 * (kk % 4) + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_addr(kt + (kk / 4) * C::SUB) + swz(tok, c), b0, b1, b2, b3);
                mma16816<KV>(sc[0], qa[kk], b0, b1);
                mma16816<KV>(sc[1], qa[kk], b2, b3);
            }
            // causal + length mask, online softmax per row (base 2)
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = kBlockSize * j + 8 * nn + 2 * tq + e;
                    sc[nn][e] = (v0 && col <= pos0) ? sc[nn][e] * p.qscale : -INFINITY;
                    sc[nn][2 + e] = (v1 && col <= pos1) ? sc[nn][2 + e] * p.qscale : -INFINITY;
                    mx0 = fmaxf(mx0, sc[nn][e]);
                    mx1 = fmaxf(mx1, sc[nn][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
            const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
            m0 = n0;
            m1 = n1;
            float pr[2][4];
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mr = e < 2 ? n0 : n1;
                    pr[nn][e] = (sc[nn][e] == -INFINITY) ? 0.f : fast_exp2(sc[nn][e] - mr);
                }
            l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
            l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
            // P = hi + lo in two 16-bit parts (lo = rn(P - hi), the difference
            // exact in fp32): a row that sees two or three tokens would
            // otherwise carry the 2^-9 rounding of a bf16 weight into its output
            uint32_t pa[4], pl[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float x = pr[k >> 1][2 * (k & 1)], y = pr[k >> 1][2 * (k & 1) + 1];
                pa[k] = pack2<KV>(x, y);
                const float2 r = unpack2(KV{}, pa[k]);
                pl[k] = pack2<KV>(x - r.x, y - r.y);
            }
            // O = O * alpha + P V (the rescale only when some running max moved;
            // the vote is warp-uniform)
            if (__any_sync(kFull, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][0] *= a0; o[nd][1] *= a0; o[nd][2] *= a1; o[nd][3] *= a1;
                }
            }
#pragma unroll
            for (int ndp = 0; ndp < D / 16; ++ndp) {
                const int tok = ((mi & 1) ? 8 : 0) + r8, c = 2 * (ndp % 4) + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(smem_addr(vt + (ndp / 4) * C::SUB) + swz(tok, c), b0, b1, b2, b3);
                mma16816<KV>(o[2 * ndp], pa, b0, b1);
                mma16816<KV>(o[2 * ndp + 1], pa, b2, b3);
                mma16816<KV>(o[2 * ndp], pl, b0, b1);
                mma16816<KV>(o[2 * ndp + 1], pl, b2, b3);
            }
        }
        // release the stage; generic-proxy writes (the zeroing) must be
        // ordered before the next asynchronous (TMA) write into it
        if (zeroed) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    if (!aborted && pb >= 0) finalize();
    }
}


__device__ __forceinline__ void mq_merge(float& M, float& den, float4& num, float m, float l,
                                         const float4& o) {
    if (m == -INFINITY) return;
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

// One CTA per (sequence, kv head, row tile): merge the pieces of every row
// (skipping tiles finished inside one range and tiles that do not exist).
template <typename KV, int D, int G, int RT>
__global__ void __launch_bounds__(256) mq_combine_kernel(const MqCombine c) {
    griddep_wait();
    griddep_launch_dependents();
    const long long sidx = blockIdx.x;
    const int b = int(sidx / ((long long)c.hkv * c.tmax));
    const int rem = int(sidx - (long long)b * c.hkv * c.tmax);
    const int kvh = rem / c.tmax, t = rem - kvh * c.tmax;
    int n, L;
    bool bad;
    seq_shape_raw(c.cu_q, c.context_lens, b, c.mb, c.max_q, n, L, bad);
    if (n == 0 || t * RT >= n * G) return;
    const int per_head = seq_units_per_head(n, L, RT, G);
    int cum = 0;
    for (int tt = 0; tt < t; ++tt) cum += tile_blocks(n, L, tt, RT, G);
    const long long U = c.ws_prefix[c.batch];
    const long long W = mq_eff_workers(U, c.workers);
    const long long uf = (long long)c.ws_prefix[b] + (long long)kvh * per_head + cum;
    const long long ul = uf + tile_blocks(n, L, t, RT, G) - 1;
    const long long wf = ((uf + 1) * W - 1) / U, wl = ((ul + 1) * W - 1) / U;
    if (wf == wl) return;
    const int rows = min(RT, n * G - t * RT);
    const int cu = c.cu_q[b];
    for (int it = threadIdx.x; it < rows * (D / 4); it += blockDim.x) {
        const int row = it / (D / 4), d4 = it - row * (D / 4);
        float M = -INFINITY, den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        for (long long w = wf; w <= wl; ++w) {
            const long long r = (sidx + w) * RT + row;
            const float2 ml = *reinterpret_cast<const float2*>(c.part_ml + r * 2);
            const float4 o = *reinterpret_cast<const float4*>(c.part_o + r * D + 4 * d4);
            mq_merge(M, den, num, ml.x, ml.y, o);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int rr = t * RT + row;
        const long long e = ((long long)(cu + rr / G) * c.hq + kvh * G + rr % G) * D + 4 * d4;
        uint32_t* out = static_cast<uint32_t*>(c.out);
        out[e / 2] = pack2<KV>(num.x * inv, num.y * inv);
        out[e / 2 + 1] = pack2<KV>(num.z * inv, num.w * inv);
    }
}

template <typename KV, typename QT, int D, int G, int NW>
struct MqImpl {
    using C = MqCfg<D, NW, Elem<KV>::bytes>;
    static cudaError_t prepare(size_t smem) {
        return cudaFuncSetAttribute(mq_split_kernel<KV, QT, D, G, NW>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    }
    static cudaError_t occupancy(int* blocks, size_t smem) {
        cudaError_t e = prepare(smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks, mq_split_kernel<KV, QT, D, G, NW>, C::NT, smem);
    }
    static cudaError_t split(const void* k, const void* v, const MqParams& p, int grid,
                             size_t smem, cudaStream_t st) {
        return launch_pdl(mq_split_kernel<KV, QT, D, G, NW>, dim3(grid), dim3(C::NT), smem, st,
                          *static_cast<const MqSrc<KV>*>(k), *static_cast<const MqSrc<KV>*>(v), p);
    }
    static cudaError_t combine(const MqCombine& c, int grid, cudaStream_t st) {
        return launch_pdl(mq_combine_kernel<QT, D, G, C::RT>, dim3(grid), dim3(256), 0, st, c);
    }
    static MqOps ops() {
        return MqOps{C::fixed_bytes(), C::RT, C::NT, prepare, occupancy, split, combine, 1,
                     Elem<KV>::bytes == 1 ? kMqSrcRaw : kMqSrcMap};
    }
};

template <typename KV, typename QT, int D, int G>
bool mq_pick_nw(int nw, MqOps* o) {
    switch (nw) {
        case 1: *o = MqImpl<KV, QT, D, G, 1>::ops(); return true;
        case 2: *o = MqImpl<KV, QT, D, G, 2>::ops(); return true;
        case 4: *o = MqImpl<KV, QT, D, G, 4>::ops(); return true;
    }
    return false;
}
template <typename KV, typename QT, int D>
bool mq_pick_g(int G, int nw, MqOps* o) {
    switch (G) {
        case 1: return mq_pick_nw<KV, QT, D, 1>(nw, o);
        case 2: return mq_pick_nw<KV, QT, D, 2>(nw, o);
        case 4: return mq_pick_nw<KV, QT, D, 4>(nw, o);
        case 8: return mq_pick_nw<KV, QT, D, 8>(nw, o);
    }
    return false;
}
template <typename KV, typename QT>
bool mq_pick_d(int D, int G, int nw, MqOps* o) {
    if (D == 128) return mq_pick_g<KV, QT, 128>(G, nw, o);
    if (D == 64) return mq_pick_g<KV, QT, 64>(G, nw, o);
    return false;
}

}  // namespace
}  // namespace pkv
