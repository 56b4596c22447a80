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
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace pkv {
namespace {

constexpr uint64_t kMqWaitNs = 4000000000ull;
constexpr int kMqMaxBatch = 4096;
constexpr float kMqLog2e = 1.4426950408889634f;

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
// 2-D tiled TMA load of box (x, y) of `tmap` into shared memory at `dst`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tmap, int x, int y,
                                            uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// Byte offset of (row r, 16-byte chunk c) inside one 16 x 128-byte sub-tile
// written by TMA with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int D, int NW>
struct MqCfg {
    // ring depth (6 stages measured slower than 4 for the 32-row variant)
    static constexpr int NS = 4;
    static constexpr int RT = 16 * NW;                 // rows per tile
    static constexpr int NT = 32 * (NW + 1);           // threads: NW consumers + producer
    static constexpr int SUB = 16 * 128;               // one 16 x 64-element sub-tile
    static constexpr int NSUB = D / 64;                // sub-tiles per K (or V) tile
    static constexpr int TILE = NSUB * SUB;
    static constexpr int STAGE = 2 * TILE;             // K then V
    static constexpr int OFF_FULL = NS * STAGE;
    static constexpr int OFF_EMPTY = OFF_FULL + NS * 8;
    static constexpr int OFF_META = OFF_EMPTY + NS * 8;   // 2 x int4 per stage
    static constexpr int OFF_SCAN = OFF_META + NS * 32;
    static constexpr int OFF_PREFIX = OFF_SCAN + 32;
    // dynamic shared memory: alignment slack + the layout above + the prefix
    static constexpr int fixed_bytes() { return 1024 + OFF_PREFIX; }
    static_assert(D == 64 || D == 128, "head_dim");
};

__device__ __forceinline__ long long mq_eff_workers(long long U, long long W) {
    const long long cap = U / 4;   // at least 4 units per range: ranges are never empty
    return cap < 1 ? 1 : (cap < W ? cap : W);
}

template <typename KV, int D, int G, int NW>
__global__ void __launch_bounds__(32 * (NW + 1))
mq_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const MqParams p) {
    using C = MqCfg<D, NW>;
    constexpr int NS = C::NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
    int4* meta = reinterpret_cast<int4*>(smem + C::OFF_META);
    int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
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
                    const int y = (blk * p.hkv + kvh) * kBlockSize;
                    unsigned char* st = smem + s * C::STAGE;
                    mbar_arrive_expect_tx(bar, C::STAGE + extra);
#pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub) {
                        tma_load_2d(smem_addr(st + sub * C::SUB), &tmk, 64 * sub, y, bar);
                        tma_load_2d(smem_addr(st + C::TILE + sub * C::SUB), &tmv, 64 * sub, y, bar);
                    }
                } else {
                    flag_status(p.status, PKV_DEV_BAD_BLOCK);
                    if (extra) mbar_arrive_expect_tx(bar, extra);
                    else mbar_arrive(bar);
                }
            }
        }
        return;
    }

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

// ------------------------------------------------- tcgen05 row-tile kernel ---
// Long query runs (prefill chunks): a CTA owns two tiles of 128 rows of one
// (sequence, kv head), rows = (query, head) pairs, and walks their visible
// tokens in chunks of 64 (four blocks) on the 5th-generation tensor cores:
//   S = Q K^T      tcgen05.mma kind::f16, M = 128, N = 64, K = D, fp32 in TMEM
//   softmax        one thread per row reads its S row from TMEM (no shuffles)
//   O += P V       tcgen05.mma, M = 128, N = D, K = 64; P from shared memory
//                  (hi + lo 16-bit parts), V read MN-major straight from its
//                  TMA tile; O stays in TMEM for the whole tile.
// Warp 0 produces (TMA of K/V chunks into NSTG stages), warp 1 issues the MMAs
// and owns the TMEM allocation, warps 2-9 run the softmax and the epilogue
// (four warps per tile, one thread per row).
// Operands in shared memory use the 128-byte swizzle (TMA writes K/V that way;
// Q and P are written by threads in the same pattern). O is rescaled only when
// a row's running maximum grows by more than 2^8 (then exactly); in between P
// is taken against the older maximum, and O and l always share it.

constexpr int kTcRows = 128;       // rows per tile (TMEM lanes)
constexpr int kTcChunk = 64;       // tokens per chunk
constexpr int kTcStages = 3;
constexpr float kTcLazy = 8.0f;    // log2 growth of the max tolerated before rescaling O

// Shared-memory matrix descriptor (tcgen05): start, leading and stride byte
// offsets in 16-byte units, descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr >> 4) & 0x3fff) | (uint64_t((lbo >> 4) & 0x3fff) << 16) |
           (uint64_t((sbo >> 4) & 0x3fff) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Instruction descriptor, kind::f16 with fp32 accumulation: operand type
// (0 fp16, 1 bf16) for A and B, B K-major (0) or N-major (1), N and M.
__device__ __forceinline__ uint32_t tc_idesc(uint32_t ab_type, uint32_t b_major, uint32_t n,
                                             uint32_t m) {
    return (1u << 4) | (ab_type << 7) | (ab_type << 10) | (b_major << 16) | ((n >> 3) << 17) |
           ((m >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on `bar` once all tcgen05 operations this thread issued have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tc_ld32(uint32_t addr, float* v) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31},"
                 " [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st32(uint32_t addr, const float* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                 "%30,%31,%32};"
                 :: "r"(addr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                    "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                    "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                    "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                    "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                    "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
                    "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                    "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
                    "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])),
                    "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                    "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
                    "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
                    "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                    "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// The two tiles (rows of tiles 2u and 2u + 1) share every K/V chunk: while
// one tile's softmax runs, the tensor core works on the other tile's S or
// P.V. Warps 2-5 are tile 0's softmax, warps 6-9 tile 1's. TMEM (512
// columns): S buffers of tile x at 128 x + 64 (c % 2), O of tile x at
// 256 + 128 x.
constexpr int kTcThreads = 64 + 2 * kTcRows;

template <int D>
struct TcCfg {
    static constexpr int NH = D / 64;
    static constexpr int HALF = kTcChunk * 128;
    static constexpr int KV_STAGE = 2 * NH * HALF;
    static constexpr int QHALF = kTcRows * 128;
    static constexpr int QTILE = NH * QHALF;
    static constexpr int PBYTES = kTcRows * kTcChunk * 2;
    static constexpr int OFF_Q = 0;                                  // tile x at OFF_Q + x QTILE
    static constexpr int OFF_KV = OFF_Q + 2 * QTILE;
    static constexpr int OFF_P = OFF_KV + kTcStages * KV_STAGE;      // tile x: hi, lo
    static constexpr int OFF_BAR = OFF_P + 4 * PBYTES;
    // kv_full[S], kv_empty[S], s_full[2 tiles][2], p_full[2], o_done[2], drain
    static constexpr int NBAR = 2 * kTcStages + 9;
    static constexpr int OFF_MASK = OFF_BAR + NBAR * 8;
    static constexpr int OFF_MISC = OFF_MASK + kTcStages * 4;
    static constexpr int BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TMEM_COLS = 512;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms");
};

template <typename KV, int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
mq_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const MqParams p) {
    using C = TcCfg<D>;
    constexpr int QPT = kTcRows / G;   // queries per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = bars + kTcStages;
    uint64_t* s_full = bars + 2 * kTcStages;          // [tile][buffer]
    uint64_t* p_full = bars + 2 * kTcStages + 4;      // [tile]
    uint64_t* o_done = bars + 2 * kTcStages + 6;      // [tile]
    uint64_t* drain = bars + 2 * kTcStages + 8;
    int* smask = reinterpret_cast<int*>(smem + C::OFF_MASK);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    griddep_wait();
    griddep_launch_dependents();
    // unit: (sequence b, kv head, tile pair u); heavier (later) pairs first
    const int tpair = (p.tmax + 1) / 2;
    const long long unit = blockIdx.x;
    const int u = tpair - 1 - int(unit % tpair);
    const int kvh = int((unit / tpair) % p.hkv);
    const int b = int(unit / ((long long)tpair * p.hkv));
    int n, L;
    bool bad;
    seq_shape_raw(p.cu_q, p.context_lens, b, p.mb, p.max_q, n, L, bad);
    if (bad && threadIdx.x == 0 && kvh == 0 && u == 0) flag_status(p.status, PKV_DEV_BAD_LENGTH);
    const int q00 = 2 * u * QPT;                           // first query of tile 0
    if (q00 >= n) return;   // the whole CTA leaves before any allocation
    const bool two = q00 + QPT < n;                         // tile 1 holds queries too
    const int cu = p.cu_q[b];
    const int q_last = min(n, q00 + (two ? 2 : 1) * QPT) - 1;
    const int pos_max = L - n + q_last;                    // last token any row may see
    const int nch = (pos_max + 1 + kTcChunk - 1) / kTcChunk;
    const int jmax = pos_max / kBlockSize;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NBAR; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_mbar_init();
        misc[1] = 0u;
    }
    for (int i = threadIdx.x; i < kTcStages * C::KV_STAGE / 16; i += kTcThreads) {
        const int s = i / (C::KV_STAGE / 16), off = i % (C::KV_STAGE / 16);
        if (off >= C::NH * C::HALF / 16)
            reinterpret_cast<uint4*>(smem + C::OFF_KV + s * C::KV_STAGE)[off] = make_uint4(0u, 0u, 0u, 0u);
    }
    // both Q tiles (query q00 + R / G, head R % G for R in 0 .. 255), zero past
    // the sequence, 128-byte-swizzled K-major
    for (int i = threadIdx.x; i < 2 * kTcRows * (D / 8); i += kTcThreads) {
        const int R = i / (D / 8), c16 = i % (D / 8);
        const int x = R / kTcRows, r = R % kTcRows;
        const int qi = q00 + R / G, h = R % G;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qi < n)
            v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                ((long long)(cu + qi) * p.hq + kvh * G + h) * D + c16 * 8);
        const int half = c16 / 8, c = c16 % 8;
        *reinterpret_cast<uint4*>(smem + C::OFF_Q + x * C::QTILE + half * C::QHALF + r * 128 +
                                  ((c ^ (r & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr((const void*)(misc + 0))), "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t role_bit) -> bool {
        if (misc[1]) return false;
        const bool ok = mbar_wait_bounded(smem_addr(bar), parity, p.wait_ns);
        if (!ok) {
            misc[1] = 1u;
            flag_status(p.status, PKV_DEV_TIMEOUT | role_bit);
        }
        return ok;
    };

    if (warp == 0) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % kTcStages;
                if (c >= kTcStages && !wait(&kv_empty[st], ((c / kTcStages) - 1) & 1, 0x400u)) break;
                int mask = 0, nl = 0;
                int blk[kTcChunk / kBlockSize];
#pragma unroll
                for (int jj = 0; jj < kTcChunk / kBlockSize; ++jj) {
                    const int j = c * (kTcChunk / kBlockSize) + jj;
                    blk[jj] = -1;
                    if (j <= jmax) {
                        const int x = __ldg(p.block_tables + (long long)b * p.mb + j);
                        if (unsigned(x) < unsigned(p.num_blocks)) {
                            blk[jj] = x;
                            mask |= 1 << jj;
                            ++nl;
                        } else {
                            flag_status(p.status, PKV_DEV_BAD_BLOCK);
                        }
                    }
                }
                smask[st] = mask;
                const uint32_t bar = smem_addr(&kv_full[st]);
                const uint32_t extra = (c == 0 && unit == p.stall_cta) ? 16u : 0u;
                if (nl || extra)
                    mbar_arrive_expect_tx(bar, uint32_t(nl * 2 * C::NH * kBlockSize * 128) + extra);
                else mbar_arrive(bar);
                ++issued;
                unsigned char* sk = smem + C::OFF_KV + st * C::KV_STAGE;
#pragma unroll
                for (int jj = 0; jj < kTcChunk / kBlockSize; ++jj) {
                    if (blk[jj] < 0) continue;
                    const int y = (blk[jj] * p.hkv + kvh) * kBlockSize;
#pragma unroll
                    for (int h = 0; h < C::NH; ++h) {
                        tma_load_2d(smem_addr(sk + h * C::HALF + jj * kBlockSize * 128), &tmk, 64 * h, y, bar);
                        tma_load_2d(smem_addr(sk + (C::NH + h) * C::HALF + jj * kBlockSize * 128), &tmv,
                                    64 * h, y, bar);
                    }
                }
            }
            // After an abort, let the copies of the last chunks issued land
            // (bounded) before the CTA may exit.
            if (misc[1])
                for (int c = max(0, issued - kTcStages); c < issued; ++c)
                    mbar_wait_bounded(smem_addr(&kv_full[c % kTcStages]), (c / kTcStages) & 1,
                                      p.wait_ns);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            const uint32_t ab = std::is_same<KV, BF16>::value ? 1u : 0u;
            const uint32_t id_s = tc_idesc(ab, 0, kTcChunk, kTcRows);
            const uint32_t id_o = tc_idesc(ab, 1, D, kTcRows);
            const uint64_t dq0 = tc_desc(smem_addr(smem + C::OFF_Q), 16, 1024);
            const uint64_t dp0 = tc_desc(smem_addr(smem + C::OFF_P), 16, 1024);
            const uint64_t dk0 = tc_desc(smem_addr(smem + C::OFF_KV), 16, 1024);
            const uint64_t dv0 = tc_desc(smem_addr(smem + C::OFF_KV + C::NH * C::HALF), C::HALF, 1024);
            auto issue_s = [&](int c, int x) {
                const uint64_t dq = dq0 + uint64_t((x * C::QTILE) >> 4);
                const uint64_t dk = dk0 + uint64_t((c % kTcStages) * (C::KV_STAGE >> 4));
                const uint32_t d = tmem + x * 2 * kTcChunk + (c & 1) * kTcChunk;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * C::QHALF + (kk % 4) * 32) >> 4;
                    const uint32_t offk = ((kk / 4) * C::HALF + (kk % 4) * 32) >> 4;
                    tc_mma(d, dq + off, dk + offk, id_s, kk > 0);
                }
                tc_commit(smem_addr(&s_full[2 * x + (c & 1)]));
            };
            auto issue_pv = [&](int c, int x) {
                const uint64_t dv = dv0 + uint64_t((c % kTcStages) * (C::KV_STAGE >> 4));
                const uint64_t dp = dp0 + uint64_t((x * 2 * C::PBYTES) >> 4);
                const uint32_t to = tmem + 4 * kTcChunk + x * 128;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kTcChunk / 16; ++kk)
                        tc_mma(to, dp + uint64_t((part * C::PBYTES + kk * 32) >> 4),
                               dv + uint64_t((kk * 16 * 128) >> 4), id_o,
                               (c > 0 || part > 0 || kk > 0) ? 1u : 0u);
                tc_commit(smem_addr(&o_done[x]));
            };
            auto finish = [&](int c) -> bool {   // P.V of chunk c for both tiles
                if (!wait(&p_full[0], c & 1, 0x800u)) return false;
                tc_fence_after();
                issue_pv(c, 0);
                if (two) {
                    if (!wait(&p_full[1], c & 1, 0x800u)) return false;
                    tc_fence_after();
                    issue_pv(c, 1);
                }
                tc_commit(smem_addr(&kv_empty[c % kTcStages]));
                return true;
            };
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                ok = wait(&kv_full[c % kTcStages], (c / kTcStages) & 1, 0x800u);
                if (!ok) break;
                tc_fence_after();
                issue_s(c, 0);
                if (two) issue_s(c, 1);
                if (c > 0) ok = finish(c - 1);
            }
            if (ok) finish(nch - 1);
            tc_commit(smem_addr(&drain[0]));
            mbar_wait_bounded(smem_addr(&drain[0]), 0, 2000000000ull);
        }
    } else {
        // -------------------------------------- softmax + epilogue, per tile ---
        const int x = (warp - 2) >> 2;                        // tile
        if (x == 0 || two) {
            const int r = 32 * (warp & 3) + lane;             // TMEM lane = row of the tile
            const uint32_t lane_addr = uint32_t(32 * (warp & 3)) << 16;
            const uint32_t tm_s = tmem + x * 2 * kTcChunk;
            const uint32_t tm_o = tmem + 4 * kTcChunk + x * 128;
            const int qi = q00 + x * QPT + r / G;
            const bool rv = qi < n;
            const int pos = L - n + qi;
            float m = -INFINITY, l = 0.f;
            unsigned char* ph = smem + C::OFF_P + x * 2 * C::PBYTES + r * 128;
            const int last_blk_tok = ((L - 1) / kBlockSize) * kBlockSize;
            const bool qpos = p.qscale > 0.f;                  // max of raw scores = max of scaled
            bool ok = true;
            for (int c = 0; c < nch; ++c) {
                const int st = c % kTcStages;
                const int tok0 = c * kTcChunk;
                if (ok) ok = __all_sync(kFull, wait(&s_full[2 * x + (c & 1)], (c >> 1) & 1, 0x1000u));
                if (ok) ok = __all_sync(kFull, wait(&kv_full[st], (c / kTcStages) & 1, 0x1000u));
                float s[kTcChunk];
                float mx = -INFINITY;
                int mask = 0;
                bool plain = false;   // warp-uniform: raw scores, every column visible
                if (ok) {
                    tc_fence_after();
                    tc_ld32(tm_s + lane_addr + (c & 1) * kTcChunk, s);
                    tc_ld32(tm_s + lane_addr + (c & 1) * kTcChunk + 32, s + 32);
                    mask = smask[st];
                    plain = __all_sync(kFull, rv && pos - tok0 >= kTcChunk - 1 &&
                                                  mask == (1 << (kTcChunk / kBlockSize)) - 1) && qpos;
                    if (plain) {
                        float mr = s[0];
#pragma unroll
                        for (int i = 1; i < kTcChunk; ++i) mr = fmaxf(mr, s[i]);
                        mx = mr * p.qscale;
                    } else {
#pragma unroll
                        for (int i = 0; i < kTcChunk; ++i) {
                            const int tok = tok0 + i;
                            const bool vis = rv && tok <= pos && ((mask >> (i / kBlockSize)) & 1);
                            s[i] = vis ? s[i] * p.qscale : -INFINITY;
                            mx = fmaxf(mx, s[i]);
                        }
                    }
                    if (c > 0) ok = __all_sync(kFull, wait(&o_done[x], (c - 1) & 1, 0x1000u));
                }
                if (ok) {
                    tc_fence_after();
                    const bool grow = mx > m + kTcLazy || (m == -INFINITY && mx > -INFINITY);
                    if (c > 0 && __any_sync(kFull, grow && m > -INFINITY)) {
                        const float a = (grow && m > -INFINITY) ? fast_exp2(m - mx) : 1.f;
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            float o[32];
                            tc_ld32(tm_o + lane_addr + c0, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= a;
                            tc_st32(tm_o + lane_addr + c0, o);
                        }
                        if (grow && m > -INFINITY) l *= a;
                    }
                    if (grow) m = mx;
                    // P = exp2(s - m) as hi + lo 16-bit parts, written swizzled (row r)
                    auto emit = [&](auto expo) {
#pragma unroll
                        for (int c16 = 0; c16 < kTcChunk / 8; ++c16) {
                            uint32_t hw[4], lw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x0 = expo(s[c16 * 8 + 2 * e]);
                                const float x1 = expo(s[c16 * 8 + 2 * e + 1]);
                                l += x0 + x1;
                                hw[e] = pack2<KV>(x0, x1);
                                const float2 rr = unpack2(KV{}, hw[e]);
                                lw[e] = pack2<KV>(x0 - rr.x, x1 - rr.y);
                            }
                            const uint32_t off = uint32_t((c16 ^ (r & 7)) << 4);
                            *reinterpret_cast<uint4*>(ph + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            *reinterpret_cast<uint4*>(ph + C::PBYTES + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        }
                    };
                    if (plain) {   // finite raw scores, m finite: one fma and one ex2 each
                        const float nm = -m, qs = p.qscale;
                        emit([&](float y) { return fast_exp2(fmaf(y, qs, nm)); });
                    } else {
                        emit([&](float y) { return y == -INFINITY ? 0.f : fast_exp2(y - m); });
                    }
                    // tile 0 zeroes V rows past the context (both tiles' P.V
                    // follow tile 0's P in the MMA thread's order)
                    if (x == 0 && last_blk_tok >= tok0 && last_blk_tok < tok0 + kTcChunk &&
                        L < last_blk_tok + kBlockSize) {
                        const int jj = (last_blk_tok - tok0) / kBlockSize;
                        if ((mask >> jj) & 1) {
                            const int r0 = L - last_blk_tok;
                            const int nrow = kBlockSize - r0;
                            unsigned char* vb = smem + C::OFF_KV + st * C::KV_STAGE + C::NH * C::HALF;
                            for (int i = r; i < nrow * C::NH * 8; i += kTcRows) {
                                const int row = i / (C::NH * 8), rem = i % (C::NH * 8);
                                const int h = rem / 8, c8 = rem % 8;
                                *reinterpret_cast<uint4*>(vb + h * C::HALF + (jj * kBlockSize + r0 + row) * 128 + c8 * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                tc_named_sync(1 + x, kTcRows);
                if (r == 0) mbar_arrive(smem_addr(&p_full[x]));
            }
            if (ok) ok = __all_sync(kFull, wait(&o_done[x], (nch - 1) & 1, 0x1000u));
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint16_t* dst = static_cast<uint16_t*>(p.out) + ((long long)(cu + qi) * p.hq + kvh * G + r % G) * D;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float o[32];
                    tc_ld32(tm_o + lane_addr + c0, o);
                    if (rv) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack2<KV>(o[2 * i] * inv, o[2 * i + 1] * inv);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            reinterpret_cast<uint4*>(dst + c0)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(C::TMEM_COLS));
}

// ---------------------------------------------------------------- combine ---
struct MqCombine {
    const float* part_o;
    const float* part_ml;
    const int32_t* ws_prefix;
    const int32_t* cu_q;
    const int32_t* context_lens;
    void* out;
    int batch, hq, hkv, mb, workers, tmax, max_q;
};

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

// ------------------------------------------------------------------- host ---
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// The cache as a 2-D tensor [rows = NB * Hkv * 16][D] of 16-bit values, read
// in 16 x 64 boxes with the 128-byte swizzle.
bool encode_cache_map(CUtensorMap* m, const void* base, bool bf16, int D, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MqOps {
    int fixed_smem, rt, threads;
    cudaError_t (*prepare)(size_t smem);
    cudaError_t (*occupancy)(int* blocks, size_t smem);
    cudaError_t (*split)(const CUtensorMap&, const CUtensorMap&, const MqParams&, int, size_t,
                         cudaStream_t);
    cudaError_t (*combine)(const MqCombine&, int, cudaStream_t);
};

template <typename KV, int D, int G, int NW>
struct MqImpl {
    using C = MqCfg<D, NW>;
    static cudaError_t prepare(size_t smem) {
        return cudaFuncSetAttribute(mq_split_kernel<KV, D, G, NW>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    }
    static cudaError_t occupancy(int* blocks, size_t smem) {
        cudaError_t e = prepare(smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mq_split_kernel<KV, D, G, NW>,
                                                             C::NT, smem);
    }
    static cudaError_t split(const CUtensorMap& k, const CUtensorMap& v, const MqParams& p,
                             int grid, size_t smem, cudaStream_t st) {
        return launch_pdl(mq_split_kernel<KV, D, G, NW>, dim3(grid), dim3(C::NT), smem, st, k, v, p);
    }
    static cudaError_t combine(const MqCombine& c, int grid, cudaStream_t st) {
        return launch_pdl(mq_combine_kernel<KV, D, G, C::RT>, dim3(grid), dim3(256), 0, st, c);
    }
    static MqOps ops() {
        return MqOps{C::fixed_bytes(), C::RT, C::NT, prepare, occupancy, split, combine};
    }
};

template <typename KV, int D, int G>
bool mq_pick_nw(int nw, MqOps* o) {
    switch (nw) {
        case 1: *o = MqImpl<KV, D, G, 1>::ops(); return true;
        case 2: *o = MqImpl<KV, D, G, 2>::ops(); return true;
        case 4: *o = MqImpl<KV, D, G, 4>::ops(); return true;
    }
    return false;
}
template <typename KV, int D>
bool mq_pick_g(int G, int nw, MqOps* o) {
    switch (G) {
        case 1: return mq_pick_nw<KV, D, 1>(nw, o);
        case 2: return mq_pick_nw<KV, D, 2>(nw, o);
        case 4: return mq_pick_nw<KV, D, 4>(nw, o);
    }
    return false;
}
template <typename KV>
bool mq_pick_d(int D, int G, int nw, MqOps* o) {
    if (D == 128) return mq_pick_g<KV, 128>(G, nw, o);
    if (D == 64) return mq_pick_g<KV, 64>(G, nw, o);
    return false;
}

// tcgen05 row-tile path: launchers by cache type, head dim and group size.
using TcLaunch = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const MqParams&, int,
                                 cudaStream_t);
template <typename KV, int D, int G>
cudaError_t tc_launch(const CUtensorMap& k, const CUtensorMap& v, const MqParams& p, int grid,
                      cudaStream_t st) {
    // two row tiles per CTA: grid counts tile pairs
    const int smem = TcCfg<D>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(mq_tc_kernel<KV, D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)grid / p.tmax;
    const int g2 = int(tiles * ((p.tmax + 1) / 2));
    return launch_pdl(mq_tc_kernel<KV, D, G>, dim3(g2), dim3(kTcThreads), size_t(smem), st, k, v, p);
}
template <typename KV, int D>
TcLaunch tc_pick_g(int G) {
    switch (G) {
        case 1: return tc_launch<KV, D, 1>;
        case 2: return tc_launch<KV, D, 2>;
        case 4: return tc_launch<KV, D, 4>;
    }
    return nullptr;
}
template <typename KV>
TcLaunch tc_pick(int D, int G) {
    if (D == 128) return tc_pick_g<KV, 128>(G);
    if (D == 64) return tc_pick_g<KV, 64>(G);
    return nullptr;
}

struct MqPlan {
    MqOps ops;
    int G, nw, tmax;
    long long workers;
    size_t smem, ws_prefix, ws_ml, ws_o, ws_total;
};

bool mq_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t mq_align256(size_t x) { return (x + 255) & ~size_t(255); }

// Checks the sizes and picks the kernel, tile height, workers and workspace.
pkv_status mq_plan(const pkv_cache_desc* c, int batch, int hq, int max_q, pkv_dtype q_dtype,
                   int num_parts, MqPlan* pl) {
    if (!c || c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (batch < 0 || hq <= 0 || hq % c->num_kv_heads || max_q <= 0 || num_parts < 0)
        return PKV_ERR_INVALID_ARG;
    if (c->kv_dtype != PKV_BF16 && c->kv_dtype != PKV_F16) return PKV_ERR_UNSUPPORTED;
    if (q_dtype != c->kv_dtype) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize || batch > kMqMaxBatch) return PKV_ERR_UNSUPPORTED;
    if ((long long)c->num_blocks * c->num_kv_heads * kBlockSize >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;
    pl->G = hq / c->num_kv_heads;
    const long long rows = (long long)max_q * pl->G;
    if (rows > (1LL << 24)) return PKV_ERR_UNSUPPORTED;
    pl->nw = rows <= 16 ? 1 : (rows <= 32 ? 2 : 4);
    const bool ok = c->kv_dtype == PKV_BF16 ? mq_pick_d<BF16>(c->head_dim, pl->G, pl->nw, &pl->ops)
                                            : mq_pick_d<F16>(c->head_dim, pl->G, pl->nw, &pl->ops);
    if (!ok) return PKV_ERR_UNSUPPORTED;
    pl->tmax = int((rows + pl->ops.rt - 1) / pl->ops.rt);
    pl->smem = size_t(pl->ops.fixed_smem) + 4 * size_t((batch < 1 ? 1 : batch) + 1);
    if (num_parts > 0) {
        pl->workers = num_parts;
    } else {
        int dev = 0, sms = 0, blocks = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            pl->ops.occupancy(&blocks, pl->smem) != cudaSuccess || blocks <= 0)
            return PKV_ERR_CUDA;
        pl->workers = (long long)sms * blocks;
    }
    const long long slots = (long long)batch * c->num_kv_heads * pl->tmax + pl->workers;
    pl->ws_prefix = 0;
    pl->ws_ml = mq_align256(sizeof(int32_t) * size_t(batch + 1));
    pl->ws_o = pl->ws_ml + mq_align256(size_t(slots) * pl->ops.rt * 2 * sizeof(float));
    pl->ws_total = pl->ws_o + mq_align256(size_t(slots) * pl->ops.rt * c->head_dim * sizeof(float));
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_multiquery_workspace_size(int32_t batch, int32_t num_q_heads,
                                                int32_t max_q_len, const pkv_cache_desc* cache,
                                                int32_t num_parts) {
    MqPlan pl;
    if (!cache) return 0;
    if (mq_plan(cache, batch, num_q_heads, max_q_len, cache->kv_dtype, num_parts, &pl) != PKV_OK)
        return 0;
    return pl.ws_total;
}

namespace {

constexpr uint64_t kTcWaitNs = 2000000000ull;

pkv_status run_multiquery(const void* q, pkv_dtype q_dtype, const int32_t* cu_q,
                          int32_t max_q_len, const void* k_cache, const void* v_cache,
                          const pkv_cache_desc* cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                          int32_t num_q_heads, float softmax_scale, void* out, void* workspace,
                          size_t workspace_bytes, int32_t num_parts, uint32_t* dev_status,
                          cudaStream_t stream, uint64_t wait_ns, int stall_cta) {
    MqPlan pl;
    pkv_status s = mq_plan(cache, batch, num_q_heads, max_q_len, q_dtype, num_parts, &pl);
    if (s != PKV_OK) return s;
    if (batch == 0) return PKV_OK;
    if (!q || !cu_q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!mq_aligned(q, 4) || !mq_aligned(out, 4) || !mq_aligned(k_cache, 16) ||
        !mq_aligned(v_cache, 16) || !mq_aligned(cu_q, 4) || !mq_aligned(block_tables, 4) ||
        !mq_aligned(context_lens, 4) || (dev_status && !mq_aligned(dev_status, 4)))
        return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || !(softmax_scale == softmax_scale) || softmax_scale > 3.0e38f ||
        softmax_scale < -3.0e38f || pl.workers > 0x7fffffffLL)
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.ws_total || !mq_aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    const long long rows = (long long)cache->num_blocks * cache->num_kv_heads * kBlockSize;
    CUtensorMap tk, tv;
    if (!encode_cache_map(&tk, k_cache, cache->kv_dtype == PKV_BF16, cache->head_dim, rows) ||
        !encode_cache_map(&tv, v_cache, cache->kv_dtype == PKV_BF16, cache->head_dim, rows))
        return PKV_ERR_CUDA;
    // Query runs that fill 128-row tiles take the tcgen05 kernel (no split,
    // no combine, no workspace); shorter ones the mma.sync kernel below.
    const TcLaunch tc = ((long long)max_q_len * pl.G >= kTcRows && mq_aligned(q, 16) &&
                         mq_aligned(out, 16))
                            ? (cache->kv_dtype == PKV_BF16 ? tc_pick<BF16>(cache->head_dim, pl.G)
                                                           : tc_pick<F16>(cache->head_dim, pl.G))
                            : nullptr;
    if (tc) {
        MqParams p;
        p.q = q; p.cu_q = cu_q; p.block_tables = block_tables; p.context_lens = context_lens;
        p.out = out; p.part_o = nullptr; p.part_ml = nullptr; p.ws_prefix = nullptr;
        p.status = dev_status;
        p.batch = batch; p.hq = num_q_heads; p.hkv = cache->num_kv_heads;
        p.mb = max_blocks_per_seq; p.num_blocks = cache->num_blocks; p.workers = 0;
        p.tmax = int(((long long)max_q_len * pl.G + kTcRows - 1) / kTcRows);
        p.max_q = max_q_len;
        p.qscale = softmax_scale * kMqLog2e;
        p.wait_ns = wait_ns < kTcWaitNs ? wait_ns : kTcWaitNs;
        p.stall_cta = stall_cta;
        const long long grid = (long long)batch * p.hkv * p.tmax;
        if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
        if (tc(tk, tv, p, int(grid), stream) != cudaSuccess) return PKV_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    }
    char* ws = static_cast<char*>(workspace);
    MqParams p;
    p.q = q; p.cu_q = cu_q; p.block_tables = block_tables; p.context_lens = context_lens;
    p.out = out;
    p.part_o = reinterpret_cast<float*>(ws + pl.ws_o);
    p.part_ml = reinterpret_cast<float*>(ws + pl.ws_ml);
    p.ws_prefix = reinterpret_cast<int32_t*>(ws + pl.ws_prefix);
    p.status = dev_status;
    p.batch = batch; p.hq = num_q_heads; p.hkv = cache->num_kv_heads; p.mb = max_blocks_per_seq;
    p.num_blocks = cache->num_blocks; p.workers = int(pl.workers); p.tmax = pl.tmax;
    p.max_q = max_q_len;
    p.qscale = softmax_scale * kMqLog2e;
    p.wait_ns = wait_ns;
    p.stall_cta = stall_cta;
    if (pl.ops.prepare(pl.smem) != cudaSuccess) return PKV_ERR_CUDA;
    if (pl.ops.split(tk, tv, p, int(pl.workers), pl.smem, stream) != cudaSuccess)
        return PKV_ERR_CUDA;
    MqCombine cb;
    cb.part_o = p.part_o; cb.part_ml = p.part_ml; cb.ws_prefix = p.ws_prefix; cb.cu_q = cu_q;
    cb.context_lens = context_lens; cb.out = out; cb.batch = batch; cb.hq = num_q_heads;
    cb.hkv = p.hkv; cb.mb = max_blocks_per_seq; cb.workers = p.workers; cb.tmax = pl.tmax;
    cb.max_q = max_q_len;
    const long long grid = (long long)batch * p.hkv * pl.tmax;
    if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    if (pl.ops.combine(cb, int(grid), stream) != cudaSuccess) return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" pkv_status pkv_multiquery_attn(const void* q, pkv_dtype q_dtype, const int32_t* cu_q,
                                          int32_t max_q_len, const void* k_cache,
                                          const void* v_cache, const pkv_cache_desc* cache,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t batch,
                                          int32_t num_q_heads, float softmax_scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t num_parts, uint32_t* dev_status,
                                          cudaStream_t stream) {
    return run_multiquery(q, q_dtype, cu_q, max_q_len, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, batch, num_q_heads, softmax_scale, out,
                          workspace, workspace_bytes, num_parts, dev_status, stream, kMqWaitNs,
                          -1);
}

// ------------------------------------------------------------- test hook ---
#include "../../include/pkv_testing.h"

extern "C" pkv_status pkv_testing_multiquery_attn_stall(
    const void* q, pkv_dtype q_dtype, const int32_t* cu_q, int32_t max_q_len, const void* k_cache,
    const void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
    float softmax_scale, void* out, void* workspace, size_t workspace_bytes, int32_t num_parts,
    uint64_t wait_limit_ns, int32_t stall_cta, uint32_t* dev_status, cudaStream_t stream) {
    if (wait_limit_ns > kMqWaitNs || stall_cta < -1) return PKV_ERR_INVALID_ARG;
    return run_multiquery(q, q_dtype, cu_q, max_q_len, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, batch, num_q_heads, softmax_scale, out,
                          workspace, workspace_bytes, num_parts, dev_status, stream, wait_limit_ns,
                          stall_cta);
}
