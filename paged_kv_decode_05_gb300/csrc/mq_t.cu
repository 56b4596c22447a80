// Multi-query attention for short query runs, over fp16 / bf16 caches and
// (head_dim 128) INT8 caches: at most 24 rows (n_b queries x g heads) per
// (sequence, kv head), the shape of
// speculative verification, where the target model scores the draft's
// tokens plus one in one batched pass (Continuous-Batching-LLM-Inference-
// Engine README, feature list "Speculative decoding"). Query i of sequence b
// sits at position L_b - n_b + i and attends to positions 0 .. L_b - n_b + i.
//
// GB300 design: the query rows sit on the N side of the MMA in tiles of 8
// columns (20 rows take 24 columns; in the 16-rows-per-warp layout of
// mq_split_kernel they take 32 MMA rows in two warps that both read every
// tile), and one warp does all the math of a unit.
// * One warp per worker: the unit stream (sequence, kv head, block) is cut
//   into equal ranges per warp, and each warp streams its range through its
//   own ring of stages, filled by 2-D TMA tensor copies of each 16-token K
//   and V tile in 64-column boxes with the 128-byte swizzle.
// * S^T[16 tokens x 8 NT rows] = K Q^T on mma.sync m16n8k16 (fp32
//   accumulate): K's A fragments come from ldmatrix, the rows' q stays in
//   registers as B fragments for the whole piece.
// * O^T[D x rows] += V^T P^T: V^T's A fragments come from ldmatrix.trans of
//   the swizzled V tile; P goes through a padded shared-memory buffer (one
//   row per query row) into B fragments, as hi + lo parts of the cache type.
// * Pieces that cross ranges leave (m, l, o) partials in the multi-query
//   workspace layout (one row tile of 8 NT rows), which the multi-query
//   combine kernel merges.
#include "mq_split.cuh"

namespace pkv {
namespace {

constexpr uint64_t kMqtDrainNs = 100000000ull;   // 100 ms per stage when draining

__host__ __device__ constexpr int mqt_align(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int NT>
struct MqtCfg {
    static constexpr int WARPS = 4;                  // worker warps per CTA, 2 CTAs per SM
    static constexpr int R = 8 * NT;                 // query rows per (sequence, kv head)
    static constexpr int SUB = kBlockSize * 128;     // one 16 x 64-element box (swizzled)
    static constexpr int NSUB = D / 64;              // boxes per K (or V) tile
    static constexpr int TILE = NSUB * SUB;
    static constexpr int STAGE = 2 * TILE;           // K then V
    static constexpr int NS = D == 128 ? 3 : 6;      // stages per warp (24 KB)
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int OFF_META = mqt_align(OFF_BAR + NS * 8, 16);   // 2 int4 per stage
    static constexpr int OFF_P = OFF_META + NS * 32;
    // P[row][token] in floats; the pitch of 20 puts the 32 lanes' stores of
    // one (n-tile, e) step in 32 different banks
    static constexpr int PS = kBlockSize + 4;
    // warp regions start 1024-byte aligned: the 128-byte swizzle repeats
    // every 8 rows, and TMA writes a swizzled box at a 1024-byte boundary
    static constexpr int WARP_BYTES = mqt_align(OFF_P + R * PS * 4, 1024);
    static_assert(STAGE % 1024 == 0, "swizzled boxes start 1024-byte aligned");
};

template <typename KV, int D, int G, int NT>
__global__ void __launch_bounds__(32 * MqtCfg<D, NT>::WARPS, 2)
mqt_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const MqParams p) {
    using C = MqtCfg<D, NT>;
    constexpr int MT = D / 16;                       // m-tiles of P.V (16 dims each)
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    int* prefix = reinterpret_cast<int*>(smem) + C::WARPS;
    griddep_wait();
    griddep_launch_dependents();
    mq_build_prefix<32 * C::WARPS>(p, reinterpret_cast<int*>(smem), prefix, C::R, G);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long U = prefix[p.batch];
    const long long W = mq_eff_workers(U, p.workers);
    const long long w = (long long)blockIdx.x * C::WARPS + warp;
    if (w >= W || U == 0) return;
    const int u0 = int(w * U / W), u1 = int((w + 1) * U / W);

    unsigned char* region =
        smem + mqt_align(4 * (C::WARPS + p.batch + 1), 1024) + warp * C::WARP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(region + C::OFF_BAR);
    int4* meta = reinterpret_cast<int4*>(region + C::OFF_META);
    float* pbuf = reinterpret_cast<float*>(region + C::OFF_P);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < C::NS; ++s) mbar_init(smem_addr(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: the units' table entries 32 at a time, one per lane;
    // lane 0 issues each unit's tile copies into its stage
    auto fetch = [&](int base, int& b, int& kvh, int& j, int& n, int& L, int& blk, int& cu) {
        const int u = base + lane;
        if (u < u1) {
            int t;   // always 0: one row tile holds all rows
            mq_decode_unit(p, prefix, u, C::R, G, b, kvh, t, j, n, L);
            blk = __ldg(p.block_tables + (long long)b * p.mb + j);
            cu = __ldg(p.cu_q + b);
        } else {
            b = kvh = j = n = L = cu = 0;
            blk = -1;
        }
    };
    int cbase = u0;
    int cb, ck, cj, cn, cL, cblk, ccu, xb, xk, xj, xn, xL, xblk, xcu;
    fetch(cbase, cb, ck, cj, cn, cL, cblk, ccu);
    fetch(cbase + 32, xb, xk, xj, xn, xL, xblk, xcu);
    auto issue = [&](int u, int s, uint32_t extra_tx) {
        int idx = u - cbase;
        if (idx >= 32) {
            cbase += 32;
            cb = xb; ck = xk; cj = xj; cn = xn; cL = xL; cblk = xblk; ccu = xcu;
            fetch(cbase + 32, xb, xk, xj, xn, xL, xblk, xcu);
            idx -= 32;
        }
        const int b = __shfl_sync(kFull, cb, idx), kvh = __shfl_sync(kFull, ck, idx);
        const int j = __shfl_sync(kFull, cj, idx), n = __shfl_sync(kFull, cn, idx);
        const int L = __shfl_sync(kFull, cL, idx), blk = __shfl_sync(kFull, cblk, idx);
        const int cu = __shfl_sync(kFull, ccu, idx);
        if (lane == 0) {
            const uint32_t bar = smem_addr(&bars[s]);
            const bool valid = unsigned(blk) < unsigned(p.num_blocks);
            const bool first = (u == u0) || (j == 0);   // first unit of a piece
            // flags: bit 0 = tiles copied, bit 1 = first unit of a piece
            meta[2 * s] = make_int4(b, kvh, j, (valid ? 1 : 0) | (first ? 2 : 0));
            meta[2 * s + 1] = make_int4(n, L, cu, 0);
            if (valid) {
                mbar_arrive_expect_tx(bar, C::STAGE + extra_tx);
                const int y = (blk * p.hkv + kvh) * kBlockSize;   // < 2^31: checked on the host
                unsigned char* st = region + s * C::STAGE;
#pragma unroll
                for (int sub = 0; sub < C::NSUB; ++sub) {
                    tma_load_2d(smem_addr(st + sub * C::SUB), &tmk, 64 * sub, y, bar);
                    tma_load_2d(smem_addr(st + C::TILE + sub * C::SUB), &tmv, 64 * sub, y, bar);
                }
            } else {
                flag_status(p.status, PKV_DEV_BAD_BLOCK);
                if (extra_tx) mbar_arrive_expect_tx(bar, extra_tx);
                else mbar_arrive(bar);
            }
        }
    };

    // ---- consumer. Lane (gq, tq) = (lane / 4, lane % 4):
    //  * S^T: rows = tokens gq, gq + 8 of the tile; columns = query rows
    //    8 nt + 2 tq + e of n-tile nt.
    //  * O^T += V^T P^T: m-tile i covers dims 16 i .. 16 i + 15; the lane
    //    accumulates dims 16 i + gq and 16 i + gq + 8 of its rows
    //    8 nt + 2 tq + e, so it keeps their softmax state.
    // Row r is query r / g, head r % g; rows past n_b g are padding.
    // ldmatrix row addresses: lane = 8 mi + r8 supplies row r8 of matrix mi.
    const int gq = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int ktok = ((mi & 1) ? 8 : 0) + r8, kch = mi >> 1;   // K: A = [tokens x dims]
    const int vtok = ((mi & 2) ? 8 : 0) + r8, vch = mi & 1;    // V^T: A = [dims x tokens]
    uint32_t qb[NT][D / 16][2];                      // q^T B fragments, rows 8 nt + gq
    float m[NT][2], lsum[NT][2];
    float oa[NT][MT][4];
    int pos[NT][2];                                  // positions of rows 8 nt + 2 tq + e (-1: padding)
    int pb = -1, pk = 0, pn = 0, pL = 0, pcu = 0, first_j = 0, last_j = 0;

    auto finalize = [&]() {
        const bool whole = first_j == 0 && last_j == (pL - 1) / kBlockSize;
        const long long slot = ((long long)pb * p.hkv + pk) * p.tmax + w;   // row tile 0
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = lsum[nt][e];
                l += __shfl_xor_sync(kFull, l, 4);
                l += __shfl_xor_sync(kFull, l, 8);
                l += __shfl_xor_sync(kFull, l, 16);
                if (pos[nt][e] < 0) continue;
                const int r = 8 * nt + 2 * tq + e;
                if (whole) {
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    const int i = r / G, h = r - (r / G) * G;
                    const long long off = ((long long)(pcu + i) * p.hq + pk * G + h) * D + gq;
#pragma unroll
                    for (int k = 0; k < MT; ++k) {
                        store_scalar(KV{}, p.out, off + 16 * k, oa[nt][k][e] * inv);
                        store_scalar(KV{}, p.out, off + 16 * k + 8, oa[nt][k][2 + e] * inv);
                    }
                } else {
                    const long long ri = slot * C::R + r;
                    float* dst = p.part_o + ri * D + gq;
#pragma unroll
                    for (int k = 0; k < MT; ++k) {
                        dst[16 * k] = oa[nt][k][e];
                        dst[16 * k + 8] = oa[nt][k][2 + e];
                    }
                    if (gq == 0)
                        *reinterpret_cast<float2*>(p.part_ml + ri * 2) = make_float2(m[nt][e], l);
                }
            }
    };

    for (int s = 0; s < C::NS; ++s)
        if (u0 + s < u1) issue(u0 + s, s, (s == 0 && w == p.stall_cta) ? 16u : 0u);
    int u_issue = (u0 + C::NS < u1) ? u0 + C::NS : u1;
    uint32_t parity = 0;
    int u = u0;
    bool aborted = false;
    int s = 0;                       // stage of unit u
    for (; u < u1; ++u, s = (s + 1 == C::NS) ? 0 : s + 1) {
        const bool got = mbar_wait_bounded(smem_addr(&bars[s]), (parity >> s) & 1u, p.wait_ns);
        if (!__all_sync(kFull, got)) {          // records where it gave up: bit 8 (consumer)
            if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT | 0x100u);
            aborted = true;
            break;
        }
        parity ^= 1u << s;
        const int4 ma = meta[2 * s], mb = meta[2 * s + 1];
        if (ma.w & 2) {  // first unit of a new piece: the rows' q, positions and state
            if (pb >= 0) finalize();
            pb = ma.x; pk = ma.y; first_j = ma.z; pn = mb.x; pL = mb.y; pcu = mb.z;
            const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int r = 8 * nt + gq;
                const bool rv = r < pn * G;
                const int i = r / G, h = r - (r / G) * G;
                // 32-bit words of dims 16 kk + 2 tq (b0) and + 8 (b1)
                const long long off = (((long long)(pcu + i) * p.hq + pk * G + h) * D) / 2 + tq;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    qb[nt][kk][0] = rv ? __ldg(q32 + off + 8 * kk) : 0u;
                    qb[nt][kk][1] = rv ? __ldg(q32 + off + 8 * kk + 4) : 0u;
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int rr = 8 * nt + 2 * tq + e;
                    pos[nt][e] = rr < pn * G ? pL - pn + rr / G : -1;
                    m[nt][e] = -INFINITY;
                    lsum[nt][e] = 0.f;
                }
#pragma unroll
                for (int i2 = 0; i2 < MT; ++i2)
                    oa[nt][i2][0] = oa[nt][i2][1] = oa[nt][i2][2] = oa[nt][i2][3] = 0.f;
            }
        }
        last_j = ma.z;

        bool zeroed = false;
        if (ma.w & 1) {
            unsigned char* kt = region + s * C::STAGE;
            unsigned char* vt = kt + C::TILE;
            const int nv = min(kBlockSize, pL - kBlockSize * ma.z);   // tokens present
            if (nv < kBlockSize) {   // stale V rows may hold NaN: P.V must read zeros there
                for (int off = lane * 16; off < (kBlockSize - nv) * 128; off += 32 * 16)
#pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub)
                        *reinterpret_cast<uint4*>(vt + sub * C::SUB + nv * 128 + off) =
                            make_uint4(0u, 0u, 0u, 0u);
                zeroed = true;
                __syncwarp();
            }
            // S^T in CH accumulator chains per n-tile (even / odd k-steps when
            // one n-tile alone would leave the MMAs a single dependent chain)
            constexpr int CH = NT == 1 ? 2 : 1;
            float acc[NT][CH][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a[4];
                ldsm_x4(smem_addr(kt + (kk / 4) * C::SUB) + swz(ktok, 2 * (kk % 4) + kch),
                        a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816<KV>(acc[nt][kk % CH], a, qb[nt][kk][0], qb[nt][kk][1]);
            }
            // causal mask (which also masks tokens past L), online softmax per
            // row in base 2, P[row][token] to shared memory
            const int tp = kBlockSize * ma.z + gq;
            bool moved = false;
            float alpha[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a0 = acc[nt][0][e], a1 = acc[nt][0][2 + e];
                    if constexpr (CH == 2) {
                        a0 += acc[nt][1][e];
                        a1 += acc[nt][1][2 + e];
                    }
                    const float s0 = (tp <= pos[nt][e]) ? a0 * p.qscale : -INFINITY;
                    const float s1 = (tp + 8 <= pos[nt][e]) ? a1 * p.qscale : -INFINITY;
                    float bm = fmaxf(s0, s1);
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
                    const float mn = fmaxf(m[nt][e], bm);
                    alpha[nt][e] = (mn == -INFINITY) ? 1.f : fast_exp2(m[nt][e] - mn);
                    moved |= alpha[nt][e] != 1.f;
                    m[nt][e] = mn;
                    const float p0 = (s0 == -INFINITY) ? 0.f : fast_exp2(s0 - mn);
                    const float p1 = (s1 == -INFINITY) ? 0.f : fast_exp2(s1 - mn);
                    lsum[nt][e] = lsum[nt][e] * alpha[nt][e] + (p0 + p1);
                    float* prow = pbuf + (8 * nt + 2 * tq + e) * C::PS;
                    prow[gq] = p0;
                    prow[gq + 8] = p1;
                }
            if (__any_sync(kFull, moved)) {   // rescale O only when some running max moved
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        oa[nt][i][0] *= alpha[nt][0]; oa[nt][i][1] *= alpha[nt][1];
                        oa[nt][i][2] *= alpha[nt][0]; oa[nt][i][3] *= alpha[nt][1];
                    }
            }
            __syncwarp();
            // P^T as the B operand of n-tile nt: column gq = row 8 nt + gq,
            // tokens 2tq, 2tq + 1 | 2tq + 8, 2tq + 9, as hi + lo parts of the
            // cache type (hi = rn(P), lo = rn(P - hi), the difference exact
            // in fp32): a weight in [0, 1] is then off by at most 2^-18 (bf16)
            // where one 16-bit P would leave up to 2^-9 |v| on a short row.
            uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float2 f = *reinterpret_cast<const float2*>(
                        pbuf + (8 * nt + gq) * C::PS + 2 * tq + 8 * k);
                    ph[nt][k] = pack2<KV>(f.x, f.y);
                    const float2 r = unpack2(KV{}, ph[nt][k]);
                    pl[nt][k] = pack2<KV>(f.x - r.x, f.y - r.y);
                }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                uint32_t va[4];
                ldsm_x4_trans(smem_addr(vt + (i / 4) * C::SUB) + swz(vtok, 2 * (i % 4) + vch),
                              va[0], va[1], va[2], va[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma16816<KV>(oa[nt][i], va, ph[nt][0], ph[nt][1]);
                    mma16816<KV>(oa[nt][i], va, pl[nt][0], pl[nt][1]);
                }
            }
        }
        // the stage goes back to the copy engine once every lane is done with
        // it; generic-proxy writes (the zeroing) are ordered before the next
        // asynchronous (TMA) write into it
        if (zeroed) fence_proxy_async_smem();
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
    for (int v = u; v < u_issue; ++v) {
        const int sv = (v - u0) % C::NS;
        mbar_wait_bounded(smem_addr(&bars[sv]), (parity >> sv) & 1u, kMqtDrainNs);
        parity ^= 1u << sv;
    }
}

// ---------------------------------------------------------------- INT8 ---
// The same layout over INT8 caches (head_dim 128: one 128-byte row of codes
// per token, one swizzled TMA box per tile). Codes c enter the fp16 MMAs as
// the exact value 1152 + c (the byte c + 128 as the low mantissa byte of
// 1024), as in the other INT8 kernels:
// * K: ldmatrix on the code tile hands lane (gq, tq) four codes of token gq
//   (and gq + 8) per 16-byte chunk, dims 16c + 4tq .. + 3; k-step c takes
//   dims 16c + 4tq + {0, 1} as the contraction indices 2tq, 2tq + 1 and
//   + {2, 3} as 2tq + 8, 2tq + 9 (a permutation of the chunk's 16 dims; q's
//   B fragments follow it). q is rounded to fp16; the bias 1152 sum_d q_d of
//   a row comes off its scores before the block's K scale.
// * V^T: ldmatrix.trans hands a lane codes (tokens 2tq, 2tq + 1) x (dims
//   2gq, 2gq + 1) of a chunk; m-tile c takes dim 16c + 2gq as row gq and
//   16c + 2gq + 1 as row gq + 8 (output dims permuted), so a lane ends up
//   with adjacent output dims. P enters as one fp16 value w = rn16(P s_v),
//   s_v the block's V scale; 1152 sum_t w_t comes off each row when the
//   piece is written. O is kept in units of 2^vexp (raised when a scale would
//   push w toward the fp16 limit), as in the decode kernel.
template <int NT>
struct MqtI8Cfg {
    static constexpr int D = 128;
    static constexpr int WARPS = 4;
    static constexpr int R = 8 * NT;
    static constexpr int TILE = kBlockSize * D;      // one swizzled box of codes
    static constexpr int STAGE = 2 * TILE;           // K then V
    static constexpr int NS = 6;                     // stages per warp (24 KB)
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int OFF_META = mqt_align(OFF_BAR + NS * 8, 16);   // 2 int4 per stage
    static constexpr int OFF_SCL = OFF_META + NS * 32;                // float2 per stage
    static constexpr int OFF_P = mqt_align(OFF_SCL + NS * 8, 16);
    static constexpr int PS = kBlockSize + 4;
    static constexpr int WARP_BYTES = mqt_align(OFF_P + R * PS * 4, 1024);
    static_assert(STAGE % 1024 == 0, "swizzled boxes start 1024-byte aligned");
};

template <typename QT, int G, int NT>
__global__ void __launch_bounds__(32 * MqtI8Cfg<NT>::WARPS, 2)
mqt_i8_split_kernel(const __grid_constant__ MqI8Map ksrc, const __grid_constant__ MqI8Map vsrc,
                    const MqParams p) {
    using C = MqtI8Cfg<NT>;
    constexpr int D = C::D;
    constexpr int MT = D / 16;                       // k-steps of S, m-tiles of P.V
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    int* prefix = reinterpret_cast<int*>(smem) + C::WARPS;
    griddep_wait();
    griddep_launch_dependents();
    mq_build_prefix<32 * C::WARPS>(p, reinterpret_cast<int*>(smem), prefix, C::R, G);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long U = prefix[p.batch];
    const long long W = mq_eff_workers(U, p.workers);
    const long long w = (long long)blockIdx.x * C::WARPS + warp;
    if (w >= W || U == 0) return;
    const int u0 = int(w * U / W), u1 = int((w + 1) * U / W);

    unsigned char* region =
        smem + mqt_align(4 * (C::WARPS + p.batch + 1), 1024) + warp * C::WARP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(region + C::OFF_BAR);
    int4* meta = reinterpret_cast<int4*>(region + C::OFF_META);
    float2* scl = reinterpret_cast<float2*>(region + C::OFF_SCL);
    float* pbuf = reinterpret_cast<float*>(region + C::OFF_P);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < C::NS; ++s) mbar_init(smem_addr(&bars[s]), 2);   // + the scales' cp.async
        fence_mbar_init();
    }
    __syncwarp();

    auto fetch = [&](int base, int& b, int& kvh, int& j, int& n, int& L, int& blk, int& cu) {
        const int u = base + lane;
        if (u < u1) {
            int t;   // always 0: one row tile holds all rows
            mq_decode_unit(p, prefix, u, C::R, G, b, kvh, t, j, n, L);
            blk = __ldg(p.block_tables + (long long)b * p.mb + j);
            cu = __ldg(p.cu_q + b);
        } else {
            b = kvh = j = n = L = cu = 0;
            blk = -1;
        }
    };
    int cbase = u0;
    int cb, ck, cj, cn, cL, cblk, ccu, xb, xk, xj, xn, xL, xblk, xcu;
    fetch(cbase, cb, ck, cj, cn, cL, cblk, ccu);
    fetch(cbase + 32, xb, xk, xj, xn, xL, xblk, xcu);
    auto issue = [&](int u, int s, uint32_t extra_tx) {
        int idx = u - cbase;
        if (idx >= 32) {
            cbase += 32;
            cb = xb; ck = xk; cj = xj; cn = xn; cL = xL; cblk = xblk; ccu = xcu;
            fetch(cbase + 32, xb, xk, xj, xn, xL, xblk, xcu);
            idx -= 32;
        }
        const int b = __shfl_sync(kFull, cb, idx), kvh = __shfl_sync(kFull, ck, idx);
        const int j = __shfl_sync(kFull, cj, idx), n = __shfl_sync(kFull, cn, idx);
        const int L = __shfl_sync(kFull, cL, idx), blk = __shfl_sync(kFull, cblk, idx);
        const int cu = __shfl_sync(kFull, ccu, idx);
        if (lane == 0) {
            const uint32_t bar = smem_addr(&bars[s]);
            const bool valid = unsigned(blk) < unsigned(p.num_blocks);
            const bool first = (u == u0) || (j == 0);
            meta[2 * s] = make_int4(b, kvh, j, (valid ? 1 : 0) | (first ? 2 : 0));
            meta[2 * s + 1] = make_int4(n, L, cu, 0);
            if (valid) {
                mbar_arrive_expect_tx(bar, C::STAGE + extra_tx);
                const int tile = blk * p.hkv + kvh;   // rows tile * 16 < 2^31: checked on the host
                unsigned char* st = region + s * C::STAGE;
                tma_load_2d(smem_addr(st), &ksrc.map, 0, tile * kBlockSize, bar);
                tma_load_2d(smem_addr(st + C::TILE), &vsrc.map, 0, tile * kBlockSize, bar);
                cp_async_4(smem_addr(&scl[s].x), ksrc.scales + tile);
                cp_async_4(smem_addr(&scl[s].y), vsrc.scales + tile);
                cp_async_arrive_noinc(bar);
            } else {
                flag_status(p.status, PKV_DEV_BAD_BLOCK);
                if (extra_tx) mbar_arrive_expect_tx(bar, extra_tx);
                else mbar_arrive(bar);
                mbar_arrive(bar);
            }
        }
    };

    const int gq = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int ltok = ((mi & 1) ? 8 : 0) + r8, lch = mi >> 1;   // ldmatrix row of matrix mi
    uint32_t qb[NT][MT][2];                          // fp16 q^T B fragments (permuted dims)
    float kb[NT][2];                                 // 1152 sum_d q_d of rows 8 nt + 2tq + e
    float m[NT][2], lsum[NT][2], pw[NT][2];
    float oa[NT][MT][4];
    int pos[NT][2];
    int vexp = 0;
    float vmul = 1.f;
    int pb = -1, pk = 0, pn = 0, pL = 0, pcu = 0, first_j = 0, last_j = 0;

    auto finalize = [&]() {
        const bool whole = first_j == 0 && last_j == (pL - 1) / kBlockSize;
        const long long slot = ((long long)pb * p.hkv + pk) * p.tmax + w;   // row tile 0
        const float up = ldexpf(1.f, vexp);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = lsum[nt][e], ws = pw[nt][e];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l += __shfl_xor_sync(kFull, l, off);
                    ws += __shfl_xor_sync(kFull, ws, off);
                }
                if (pos[nt][e] < 0) continue;
                const int r = 8 * nt + 2 * tq + e;
                const float cb = 1152.f * ws;
                if (whole) {
                    const float inv = l > 0.f ? up / l : 0.f;
                    const int i = r / G, h = r - (r / G) * G;
                    const long long off = ((long long)(pcu + i) * p.hq + pk * G + h) * D + 2 * gq;
                    uint32_t* dst = static_cast<uint32_t*>(p.out);
#pragma unroll
                    for (int c = 0; c < MT; ++c)
                        dst[(off + 16 * c) / 2] = pack2<QT>((oa[nt][c][e] - cb) * inv,
                                                            (oa[nt][c][2 + e] - cb) * inv);
                } else {
                    const long long ri = slot * C::R + r;
                    float* dst = p.part_o + ri * D + 2 * gq;
#pragma unroll
                    for (int c = 0; c < MT; ++c)
                        *reinterpret_cast<float2*>(dst + 16 * c) =
                            make_float2((oa[nt][c][e] - cb) * up, (oa[nt][c][2 + e] - cb) * up);
                    if (gq == 0)
                        *reinterpret_cast<float2*>(p.part_ml + ri * 2) = make_float2(m[nt][e], l);
                }
            }
    };

    for (int s = 0; s < C::NS; ++s)
        if (u0 + s < u1) issue(u0 + s, s, (s == 0 && w == p.stall_cta) ? 16u : 0u);
    int u_issue = (u0 + C::NS < u1) ? u0 + C::NS : u1;
    uint32_t parity = 0;
    int u = u0;
    bool aborted = false;
    int s = 0;
    for (; u < u1; ++u, s = (s + 1 == C::NS) ? 0 : s + 1) {
        const bool got = mbar_wait_bounded(smem_addr(&bars[s]), (parity >> s) & 1u, p.wait_ns);
        if (!__all_sync(kFull, got)) {          // records where it gave up: bit 8 (consumer)
            if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT | 0x100u);
            aborted = true;
            break;
        }
        parity ^= 1u << s;
        const int4 ma = meta[2 * s], mb = meta[2 * s + 1];
        if (ma.w & 2) {  // first unit of a new piece: the rows' q, biases, positions, state
            if (pb >= 0) finalize();
            pb = ma.x; pk = ma.y; first_j = ma.z; pn = mb.x; pL = mb.y; pcu = mb.z;
            const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int r = 8 * nt + gq;
                const bool rv = r < pn * G;
                const int i = r / G, h = r - (r / G) * G;
                // 32-bit words of dims 16 c + 4 tq + {0, 1} and + {2, 3}
                const long long off = (((long long)(pcu + i) * p.hq + pk * G + h) * D) / 2 + 2 * tq;
                float qs = 0.f;
#pragma unroll
                for (int c = 0; c < MT; ++c) {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 f = unpack2(QT{}, rv ? __ldg(q32 + off + 8 * c + k) : 0u);
                        qb[nt][c][k] = pack2<F16>(f.x, f.y);
                        const float2 r16 = unpack2(F16{}, qb[nt][c][k]);   // what the MMAs multiply
                        qs += r16.x + r16.y;
                    }
                }
                qs += __shfl_xor_sync(kFull, qs, 1);
                qs += __shfl_xor_sync(kFull, qs, 2);
#pragma unroll
                for (int e = 0; e < 2; ++e) {   // row 2tq + e lives in lanes 4 (2tq + e) + [0, 4)
                    kb[nt][e] = 1152.f * __shfl_sync(kFull, qs, (8 * tq + 4 * e) & 31);
                    const int rr = 8 * nt + 2 * tq + e;
                    pos[nt][e] = rr < pn * G ? pL - pn + rr / G : -1;
                    m[nt][e] = -INFINITY;
                    lsum[nt][e] = 0.f;
                    pw[nt][e] = 0.f;
                }
#pragma unroll
                for (int c = 0; c < MT; ++c) oa[nt][c][0] = oa[nt][c][1] = oa[nt][c][2] = oa[nt][c][3] = 0.f;
            }
            vexp = 0;
            vmul = 1.f;
        }
        last_j = ma.z;

        if (ma.w & 1) {
            const unsigned char* kt = region + s * C::STAGE;
            const unsigned char* vt = kt + C::TILE;
            const float2 sc = scl[s];
            float vsc = sc.y;
            if (vsc * vmul >= 16384.f) {   // warp-uniform; raise vexp, rescale O exactly
                int ex;
                frexpf(vsc, &ex);          // vsc < 2^ex
                const int nexp = ex - 14;
                const float r = ldexpf(1.f, vexp - nexp);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int c = 0; c < MT; ++c) {
                        oa[nt][c][0] *= r; oa[nt][c][1] *= r; oa[nt][c][2] *= r; oa[nt][c][3] *= r;
                    }
                    pw[nt][0] *= r; pw[nt][1] *= r;
                }
                vexp = nexp;
                vmul = ldexpf(1.f, -nexp);
            }
            vsc *= vmul;
            // S^T: one accumulator chain per n-tile (NT chains interleave)
            constexpr int CH = NT == 1 ? 2 : 1;
            float acc[NT][CH][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
#pragma unroll
            for (int cp = 0; cp < MT / 2; ++cp) {   // chunks 2cp, 2cp + 1
                uint32_t r[4];   // (token gq | gq + 8) x (chunk 2cp | 2cp + 1)
                ldsm_x4(smem_addr(kt) + swz(ltok, 2 * cp + lch), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = 2 * cp + h;
                    const uint32_t u0 = r[2 * h] ^ 0x80808080u, u1 = r[2 * h + 1] ^ 0x80808080u;
                    const uint32_t a0 = i8x2_biased_h2(u0, 0x4140), a1 = i8x2_biased_h2(u1, 0x4140);
                    const uint32_t a2 = i8x2_biased_h2(u0, 0x4342), a3 = i8x2_biased_h2(u1, 0x4342);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_16816_f16(acc[nt][c % CH], a0, a1, a2, a3, qb[nt][c][0], qb[nt][c][1]);
                }
            }
            // causal mask, online softmax per row, w = rn16(P s_v) to shared memory
            const float sk = p.qscale * sc.x;
            const int tp = kBlockSize * ma.z + gq;
            bool moved = false;
            float alpha[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a0 = acc[nt][0][e], a1 = acc[nt][0][2 + e];
                    if constexpr (CH == 2) {
                        a0 += acc[nt][1][e];
                        a1 += acc[nt][1][2 + e];
                    }
                    const float s0 = (tp <= pos[nt][e]) ? (a0 - kb[nt][e]) * sk : -INFINITY;
                    const float s1 = (tp + 8 <= pos[nt][e]) ? (a1 - kb[nt][e]) * sk : -INFINITY;
                    float bm = fmaxf(s0, s1);
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
                    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
                    const float mn = fmaxf(m[nt][e], bm);
                    alpha[nt][e] = (mn == -INFINITY) ? 1.f : fast_exp2(m[nt][e] - mn);
                    moved |= alpha[nt][e] != 1.f;
                    m[nt][e] = mn;
                    const float p0 = (s0 == -INFINITY) ? 0.f : fast_exp2(s0 - mn);
                    const float p1 = (s1 == -INFINITY) ? 0.f : fast_exp2(s1 - mn);
                    lsum[nt][e] = lsum[nt][e] * alpha[nt][e] + (p0 + p1);
                    // the weights as the MMA will take them, so that the bias sum
                    // uses exactly the values multiplied
                    const float2 wr = __half22float2(__floats2half2_rn(p0 * vsc, p1 * vsc));
                    pw[nt][e] = fmaf(pw[nt][e], alpha[nt][e], wr.x + wr.y);
                    float* prow = pbuf + (8 * nt + 2 * tq + e) * C::PS;
                    prow[gq] = wr.x;
                    prow[gq + 8] = wr.y;
                }
            if (__any_sync(kFull, moved)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < MT; ++c) {
                        oa[nt][c][0] *= alpha[nt][0]; oa[nt][c][1] *= alpha[nt][1];
                        oa[nt][c][2] *= alpha[nt][0]; oa[nt][c][3] *= alpha[nt][1];
                    }
            }
            __syncwarp();
            // W^T B fragments of n-tile nt: column gq = row 8 nt + gq, tokens
            // 2tq, 2tq + 1 | 2tq + 8, 2tq + 9 (fp16-exact values)
            uint32_t pf[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float2 f = *reinterpret_cast<const float2*>(
                        pbuf + (8 * nt + gq) * C::PS + 2 * tq + 8 * k);
                    pf[nt][k] = pack2<F16>(f.x, f.y);
                }
            // V^T A fragments, two m-tiles per ldmatrix.trans; codes of tokens
            // past the context are finite and their weights exactly 0
#pragma unroll
            for (int cp = 0; cp < MT / 2; ++cp) {
                uint32_t r[4];   // (tokens 0-7 | 8-15) x (chunk 2cp | 2cp + 1)
                ldsm_x4_trans(smem_addr(vt) + swz(ltok, 2 * cp + lch), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = 2 * cp + h;
                    const uint32_t x = r[2 * h] ^ 0x80808080u, y = r[2 * h + 1] ^ 0x80808080u;
                    const uint32_t a0 = i8x2_biased_h2(x, 0x4240), a1 = i8x2_biased_h2(x, 0x4341);
                    const uint32_t a2 = i8x2_biased_h2(y, 0x4240), a3 = i8x2_biased_h2(y, 0x4341);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_16816_f16(oa[nt][c], a0, a1, a2, a3, pf[nt][0], pf[nt][1]);
                }
            }
        }
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
    for (int v = u; v < u_issue; ++v) {
        const int sv = (v - u0) % C::NS;
        mbar_wait_bounded(smem_addr(&bars[sv]), (parity >> sv) & 1u, kMqtDrainNs);
        parity ^= 1u << sv;
    }
}

// ------------------------------------------------------------------- host ---
template <typename KV, int D, int G, int NT>
struct MqtImpl {
    using C = MqtCfg<D, NT>;
    static cudaError_t prepare(size_t smem) {
        return cudaFuncSetAttribute(mqt_split_kernel<KV, D, G, NT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    }
    static cudaError_t occupancy(int* blocks, size_t smem) {
        cudaError_t e = prepare(smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks, mqt_split_kernel<KV, D, G, NT>, 32 * C::WARPS, smem);
    }
    static cudaError_t split(const void* k, const void* v, const MqParams& p, int grid,
                             size_t smem, cudaStream_t st) {
        return launch_pdl(mqt_split_kernel<KV, D, G, NT>, dim3(grid), dim3(32 * C::WARPS), smem,
                          st, *static_cast<const CUtensorMap*>(k),
                          *static_cast<const CUtensorMap*>(v), p);
    }
    static cudaError_t combine(const MqCombine& c, int grid, cudaStream_t st) {
        return launch_pdl(mq_combine_kernel<KV, D, G, C::R>, dim3(grid), dim3(256), 0, st, c);
    }
    static MqOps ops() {
        // dynamic shared memory: 1024-byte alignment slack, scan scratch and
        // prefix (the planner adds 4 (batch + 1) bytes) rounded up to 1024,
        // the warps' regions
        return MqOps{C::WARPS * C::WARP_BYTES + 2048 + 4 * C::WARPS, C::R, 32 * C::WARPS,
                     prepare, occupancy, split, combine, C::WARPS, kMqSrcMap};
    }
};

template <typename QT, int G, int NT>
struct MqtI8Impl {
    using C = MqtI8Cfg<NT>;
    static cudaError_t prepare(size_t smem) {
        return cudaFuncSetAttribute(mqt_i8_split_kernel<QT, G, NT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    }
    static cudaError_t occupancy(int* blocks, size_t smem) {
        cudaError_t e = prepare(smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks, mqt_i8_split_kernel<QT, G, NT>, 32 * C::WARPS, smem);
    }
    static cudaError_t split(const void* k, const void* v, const MqParams& p, int grid,
                             size_t smem, cudaStream_t st) {
        return launch_pdl(mqt_i8_split_kernel<QT, G, NT>, dim3(grid), dim3(32 * C::WARPS), smem,
                          st, *static_cast<const MqI8Map*>(k), *static_cast<const MqI8Map*>(v), p);
    }
    static cudaError_t combine(const MqCombine& c, int grid, cudaStream_t st) {
        return launch_pdl(mq_combine_kernel<QT, C::D, G, C::R>, dim3(grid), dim3(256), 0, st, c);
    }
    static MqOps ops() {
        return MqOps{C::WARPS * C::WARP_BYTES + 2048 + 4 * C::WARPS, C::R, 32 * C::WARPS,
                     prepare, occupancy, split, combine, C::WARPS, kMqSrcI8Map};
    }
};

template <typename QT, int G>
bool mqt_i8_pick_nt(int nt, MqOps* o) {
    switch (nt) {
        case 1: *o = MqtI8Impl<QT, G, 1>::ops(); return true;
        case 2: *o = MqtI8Impl<QT, G, 2>::ops(); return true;
        case 3: *o = MqtI8Impl<QT, G, 3>::ops(); return true;
    }
    return false;
}
template <typename QT>
bool mqt_i8_pick_g(int G, int nt, MqOps* o) {
    switch (G) {
        case 1: return mqt_i8_pick_nt<QT, 1>(nt, o);
        case 2: return mqt_i8_pick_nt<QT, 2>(nt, o);
        case 4: return mqt_i8_pick_nt<QT, 4>(nt, o);
        case 8: return mqt_i8_pick_nt<QT, 8>(nt, o);
    }
    return false;
}

template <typename KV, int D, int G>
bool mqt_pick_nt(int nt, MqOps* o) {
    switch (nt) {
        case 1: *o = MqtImpl<KV, D, G, 1>::ops(); return true;
        case 2: *o = MqtImpl<KV, D, G, 2>::ops(); return true;
        case 3: *o = MqtImpl<KV, D, G, 3>::ops(); return true;
    }
    return false;
}
template <typename KV, int D>
bool mqt_pick_g(int G, int nt, MqOps* o) {
    switch (G) {
        case 1: return mqt_pick_nt<KV, D, 1>(nt, o);
        case 2: return mqt_pick_nt<KV, D, 2>(nt, o);
        case 4: return mqt_pick_nt<KV, D, 4>(nt, o);
        case 8: return mqt_pick_nt<KV, D, 8>(nt, o);
    }
    return false;
}
template <typename KV>
bool mqt_pick_d(int D, int G, int nt, MqOps* o) {
    if (D == 128) return mqt_pick_g<KV, 128>(G, nt, o);
    if (D == 64) return mqt_pick_g<KV, 64>(G, nt, o);
    return false;
}

}  // namespace

bool mqt_pick(pkv_dtype kv_dtype, pkv_dtype q_dtype, int D, int G, int nt, MqOps* o) {
    if (kv_dtype == PKV_BF16) return mqt_pick_d<BF16>(D, G, nt, o);
    if (kv_dtype == PKV_F16) return mqt_pick_d<F16>(D, G, nt, o);
    if (kv_dtype == PKV_I8 && D == 128) {
        if (q_dtype == PKV_BF16) return mqt_i8_pick_g<BF16>(G, nt, o);
        if (q_dtype == PKV_F16) return mqt_i8_pick_g<F16>(G, nt, o);
    }
    return false;
}

}  // namespace pkv
