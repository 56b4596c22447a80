// Multi-query attention over fp16 / bf16 caches for short query runs: at most
// 24 rows (n_b queries x g heads) per (sequence, kv head), the shape of
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
                     prepare, occupancy, split, combine, C::WARPS, false};
    }
};

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

bool mqt_pick(pkv_dtype kv_dtype, int D, int G, int nt, MqOps* o) {
    if (kv_dtype == PKV_BF16) return mqt_pick_d<BF16>(D, G, nt, o);
    if (kv_dtype == PKV_F16) return mqt_pick_d<F16>(D, G, nt, o);
    return false;
}

}  // namespace pkv
