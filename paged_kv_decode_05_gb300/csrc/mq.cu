// Multi-query paged attention: the tcgen05 kernel for long query runs and
// the host side of pkv_multiquery_attn (the mma.sync split kernel and its
// combine live in mq_split.cuh).
#include <cuda.h>

#include <mutex>

#include "mq_split.cuh"

namespace pkv {
namespace {

// ------------------------------------------------- tcgen05 row-tile kernel ---
// Long query runs (prefill chunks): a CTA owns two tiles of 128 rows of one
// (sequence, kv head), rows = (query, head) pairs, and walks their visible
// tokens in chunks of 64 (four blocks) on the 5th-generation tensor cores:
//   S = Q K^T      tcgen05.mma kind::f16, M = 128, N = 64, K = D, fp32 in TMEM
//   softmax        one thread per row reads its S row from TMEM (no shuffles)
//   O += P V       tcgen05.mma, M = 128, N = D, K = 64; P from tensor memory
//                  (hi + lo 16-bit parts, written by the softmax over its own
//                  S buffer), V read MN-major straight from its TMA tile; O
//                  stays in TMEM for the whole tile.
// Warp 0 produces (TMA of K/V chunks into NSTG stages), warp 1 issues the MMAs
// and owns the TMEM allocation, warps 2-9 run the softmax and the epilogue
// (four warps per tile, one thread per row).
// Operands in shared memory use the 128-byte swizzle (TMA writes K/V that way;
// Q is written by threads in the same pattern). O is rescaled only when
// a row's running maximum grows by more than 2^8 (then exactly); in between P
// is taken against the older maximum, and O and l always share it.

constexpr int kTcRows = 128;       // rows per tile (TMEM lanes)
constexpr int kTcChunk = 64;       // tokens per chunk
constexpr int kTcStages = 5;
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
// 64 consecutive fp32 columns of this thread's TMEM lane, one wait.
__device__ __forceinline__ void tc_ld64(uint32_t addr, float* v) {
    uint32_t r[64];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,"
                 "%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                   "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                   "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                   "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
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
// 16 consecutive 32-bit columns of this thread's TMEM lane, no wait (the
// caller waits once with tc_wait_st).
__device__ __forceinline__ void tc_st16(uint32_t addr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15,%16};"
                 :: "r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
                    "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// d (TMEM) += a (TMEM: M rows in lanes, K 16-bit values packed two per
// column) * b (shared-memory descriptor).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void tc_named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// The two tiles (rows of tiles 2u and 2u + 1) share every K/V chunk: while
// one tile's softmax runs, the tensor core works on the other tile's S or
// P.V. Warps 2-5 are tile 0's softmax, warps 6-9 tile 1's. TMEM (512
// columns): S buffers of tile x at 128 x + 64 (c % 2), O of tile x at
// 256 + 128 x. P of chunk c replaces S of chunk c in its buffer (hi in the
// first 32 columns, lo in the next 32, two 16-bit values per column): the
// MMAs of a thread run in issue order, so the P.V of chunk c reads it before
// the S of chunk c + 2 overwrites the buffer, and the softmax of chunk c
// writes it while the P.V of chunk c - 1 still runs (it waits for that P.V
// only before touching O).
constexpr int kTcThreads = 64 + 2 * kTcRows;

template <int D>
struct TcCfg {
    static constexpr int NH = D / 64;
    static constexpr int HALF = kTcChunk * 128;
    static constexpr int KV_STAGE = 2 * NH * HALF;
    static constexpr int QHALF = kTcRows * 128;
    static constexpr int QTILE = NH * QHALF;
    static constexpr int OFF_Q = 0;                                  // tile x at OFF_Q + x QTILE
    static constexpr int OFF_KV = OFF_Q + 2 * QTILE;
    static constexpr int OFF_BAR = OFF_KV + kTcStages * KV_STAGE;
    // kv_full[S], kv_empty[S], s_full[2 tiles][2], p_full[2], o_done[2], drain
    static constexpr int NBAR = 2 * kTcStages + 9;
    static constexpr int OFF_MASK = OFF_BAR + NBAR * 8;
    static constexpr int OFF_MISC = OFF_MASK + kTcStages * 4;
    static constexpr int BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TMEM_COLS = 512;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(OFF_KV % 1024 == 0, "swizzle atoms");
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
                // P of chunk c (hi at columns 0-31, lo at 32-63 of its S buffer)
                const uint32_t tp = tmem + x * 2 * kTcChunk + (c & 1) * kTcChunk;
                const uint32_t to = tmem + 4 * kTcChunk + x * 128;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kTcChunk / 16; ++kk)
                        tc_mma_ts(to, tp + part * (kTcChunk / 2) + kk * 8,
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
                    tc_ld64(tm_s + lane_addr + (c & 1) * kTcChunk, s);
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
                }
                if (ok) {
                    const bool grow = mx > m + kTcLazy || (m == -INFINITY && mx > -INFINITY);
                    const bool rescale = c > 0 && __any_sync(kFull, grow && m > -INFINITY);
                    const float a = (grow && m > -INFINITY) ? fast_exp2(m - mx) : 1.f;
                    if (grow && m > -INFINITY) l *= a;
                    if (grow) m = mx;
                    // P = exp2(s - m) as hi + lo 16-bit parts, packed two per
                    // column into this chunk's S buffer (its own TMEM lane), where
                    // the P.V MMAs take it as their A operand
                    const uint32_t tp = tm_s + lane_addr + (c & 1) * kTcChunk;
                    auto emit = [&](auto expo) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t hw[16], lw[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float x0 = expo(s[32 * h + 2 * e]);
                                const float x1 = expo(s[32 * h + 2 * e + 1]);
                                l += x0 + x1;
                                hw[e] = pack2<KV>(x0, x1);
                                const float2 rr = unpack2(KV{}, hw[e]);
                                lw[e] = pack2<KV>(x0 - rr.x, x1 - rr.y);
                            }
                            tc_st16(tp + 16 * h, hw);
                            tc_st16(tp + kTcChunk / 2 + 16 * h, lw);
                        }
                    };
                    if (plain) {   // finite raw scores, m finite: one fma and one ex2 each
                        const float nm = -m, qs = p.qscale;
                        emit([&](float y) { return fast_exp2(fmaf(y, qs, nm)); });
                    } else {
                        emit([&](float y) { return y == -INFINITY ? 0.f : fast_exp2(y - m); });
                    }
                    tc_wait_st();
                    // O may be touched only once the previous chunk's P.V is done
                    if (c > 0) ok = __all_sync(kFull, wait(&o_done[x], (c - 1) & 1, 0x1000u));
                    if (ok && rescale) {
                        tc_fence_after();
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            float o[32];
                            tc_ld32(tm_o + lane_addr + c0, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= a;
                            tc_st32(tm_o + lane_addr + c0, o);
                        }
                    }
                    // tile 0 zeroes V rows past the context (both tiles' P.V
                    // follow tile 0's P in the MMA thread's order)
                    if (ok && x == 0 && last_blk_tok >= tok0 && last_blk_tok < tok0 + kTcChunk &&
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

// INT8 cache [rows, 128] of byte codes as 16 x 128-byte boxes, 128-byte swizzle.
bool encode_i8_map(CUtensorMap* m, const void* base, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, cuuint64_t(rows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 16};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
        case 8: return tc_launch<KV, D, 8>;
    }
    return nullptr;
}
template <typename KV>
TcLaunch tc_pick(int D, int G) {
    if (D == 128) return tc_pick_g<KV, 128>(G);
    if (D == 64) return tc_pick_g<KV, 64>(G);
    return nullptr;
}

// Query rows per (sequence, kv head) up to which fp16 / bf16 caches take the
// short-run kernel (mq_t.cu).
constexpr long long kMqtMaxRows = 24;

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
    if (c->kv_dtype != PKV_BF16 && c->kv_dtype != PKV_F16 && c->kv_dtype != PKV_I8)
        return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_BF16 && q_dtype != PKV_F16) return PKV_ERR_INVALID_ARG;
    if (c->kv_dtype != PKV_I8 && q_dtype != c->kv_dtype) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize || batch > kMqMaxBatch) return PKV_ERR_UNSUPPORTED;
    if ((long long)c->num_blocks * c->num_kv_heads * kBlockSize >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;
    pl->G = hq / c->num_kv_heads;
    const long long rows = (long long)max_q * pl->G;
    if (rows > (1LL << 24)) return PKV_ERR_UNSUPPORTED;
    pl->nw = rows <= 16 ? 1 : (rows <= 32 ? 2 : 4);
    // short runs: rows on the MMA's N side, a warp per worker (INT8: head_dim 128)
    bool ok = rows <= kMqtMaxRows &&
              mqt_pick(c->kv_dtype, q_dtype, c->head_dim, pl->G, int((rows + 7) / 8), &pl->ops);
    if (!ok && c->kv_dtype == PKV_I8)
        ok = mq_pick_i8(q_dtype, c->head_dim, pl->G, pl->nw, &pl->ops);
    else if (!ok)
        ok = c->kv_dtype == PKV_BF16 ? mq_pick_d<BF16, BF16>(c->head_dim, pl->G, pl->nw, &pl->ops)
                                     : mq_pick_d<F16, F16>(c->head_dim, pl->G, pl->nw, &pl->ops);
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
        pl->workers = (long long)sms * blocks * pl->ops.wpc;
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
    const pkv_dtype qd = cache->kv_dtype == PKV_I8 ? PKV_BF16 : cache->kv_dtype;   // same sizes
    if (mq_plan(cache, batch, num_q_heads, max_q_len, qd, num_parts, &pl) != PKV_OK) return 0;
    return pl.ws_total;
}

namespace {

constexpr uint64_t kTcWaitNs = 2000000000ull;

// The tcgen05 launcher that serves runs of max_q rows per query head group
// over this cache (16-bit caches, rows filling 128-row tiles), or nullptr;
// q and out must also be 16-byte aligned.
TcLaunch tc_for(const pkv_cache_desc* cache, int max_q, int G) {
    if (cache->kv_dtype == PKV_I8 || (long long)max_q * G < kTcRows) return nullptr;
    return cache->kv_dtype == PKV_BF16 ? tc_pick<BF16>(cache->head_dim, G)
                                       : tc_pick<F16>(cache->head_dim, G);
}

pkv_status run_multiquery(const void* q, pkv_dtype q_dtype, const int32_t* cu_q,
                          int32_t max_q_len, const void* k_cache, const void* v_cache,
                          const float* k_scales, const float* v_scales,
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
    const bool i8 = cache->kv_dtype == PKV_I8;
    if (i8 && (!k_scales || !v_scales || !mq_aligned(k_scales, 4) || !mq_aligned(v_scales, 4) ||
               !mq_aligned(q, 16)))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.ws_total || !mq_aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    const long long rows = (long long)cache->num_blocks * cache->num_kv_heads * kBlockSize;
    // 16-bit tiles through tensor maps; INT8 tiles through tensor maps of the
    // codes (short-run kernel) or 1-D bulk copies (the 32-row kernel)
    CUtensorMap tk = {}, tv = {};
    if (pl.ops.src == kMqSrcMap &&
        (!encode_cache_map(&tk, k_cache, cache->kv_dtype == PKV_BF16, cache->head_dim, rows) ||
         !encode_cache_map(&tv, v_cache, cache->kv_dtype == PKV_BF16, cache->head_dim, rows)))
        return PKV_ERR_CUDA;
    MqI8Map mk = {}, mv = {};
    if (pl.ops.src == kMqSrcI8Map) {
        if (!encode_i8_map(&mk.map, k_cache, rows) || !encode_i8_map(&mv.map, v_cache, rows))
            return PKV_ERR_CUDA;
        mk.scales = k_scales;
        mv.scales = v_scales;
    }
    // Query runs of 16-bit caches that fill 128-row tiles take the tcgen05
    // kernel (no split, no combine, no workspace); shorter runs, and every run
    // over an INT8 cache, the mma.sync kernel below.
    const TcLaunch tc = mq_aligned(q, 16) && mq_aligned(out, 16)
                            ? tc_for(cache, max_q_len, pl.G) : nullptr;
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
    const MqI8Src ik{k_cache, k_scales}, iv{v_cache, v_scales};
    const void* ks = pl.ops.src == kMqSrcRaw ? static_cast<const void*>(&ik)
                     : pl.ops.src == kMqSrcI8Map ? static_cast<const void*>(&mk)
                                                 : static_cast<const void*>(&tk);
    const void* vs = pl.ops.src == kMqSrcRaw ? static_cast<const void*>(&iv)
                     : pl.ops.src == kMqSrcI8Map ? static_cast<const void*>(&mv)
                                                 : static_cast<const void*>(&tv);
    const long long ctas = (pl.workers + pl.ops.wpc - 1) / pl.ops.wpc;
    if (pl.ops.split(ks, vs, p, int(ctas), pl.smem, stream) != cudaSuccess)
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
                                          const void* v_cache, const float* k_scales,
                                          const float* v_scales, const pkv_cache_desc* cache,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t batch,
                                          int32_t num_q_heads, float softmax_scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t num_parts, uint32_t* dev_status,
                                          cudaStream_t stream) {
    return run_multiquery(q, q_dtype, cu_q, max_q_len, k_cache, v_cache, k_scales, v_scales,
                          cache, block_tables, max_blocks_per_seq, context_lens, batch,
                          num_q_heads, softmax_scale, out, workspace, workspace_bytes, num_parts,
                          dev_status, stream, kMqWaitNs, -1);
}

// ------------------------------------------------------------- test hook ---
#include "../../include/pkv_testing.h"

extern "C" pkv_status pkv_testing_multiquery_kernel(int32_t batch, int32_t num_q_heads,
                                                    int32_t max_q_len, const pkv_cache_desc* cache,
                                                    pkv_dtype q_dtype, int32_t num_parts,
                                                    int32_t* kernel, int32_t* rows_per_tile) {
    if (!kernel || !rows_per_tile || num_parts <= 0) return PKV_ERR_INVALID_ARG;
    MqPlan pl;
    const pkv_status s = mq_plan(cache, batch, num_q_heads, max_q_len, q_dtype, num_parts, &pl);
    if (s != PKV_OK) return s;
    if (tc_for(cache, max_q_len, pl.G)) {
        *kernel = PKV_TESTING_MQ_TCGEN05;
        *rows_per_tile = kTcRows;
        return PKV_OK;
    }
    *kernel = pl.ops.src == kMqSrcI8Map ? PKV_TESTING_MQ_SHORT_I8
              : pl.ops.wpc > 1          ? PKV_TESTING_MQ_SHORT
                                        : PKV_TESTING_MQ_ROWS16;
    *rows_per_tile = pl.ops.rt;
    return PKV_OK;
}

extern "C" pkv_status pkv_testing_multiquery_attn_stall(
    const void* q, pkv_dtype q_dtype, const int32_t* cu_q, int32_t max_q_len, const void* k_cache,
    const void* v_cache, const float* k_scales, const float* v_scales,
    const pkv_cache_desc* cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
    float softmax_scale, void* out, void* workspace, size_t workspace_bytes, int32_t num_parts,
    uint64_t wait_limit_ns, int32_t stall_cta, uint32_t* dev_status, cudaStream_t stream) {
    if (wait_limit_ns > kMqWaitNs || stall_cta < -1) return PKV_ERR_INVALID_ARG;
    return run_multiquery(q, q_dtype, cu_q, max_q_len, k_cache, v_cache, k_scales, v_scales,
                          cache, block_tables, max_blocks_per_seq, context_lens, batch,
                          num_q_heads, softmax_scale, out, workspace, workspace_bytes, num_parts,
                          dev_status, stream, wait_limit_ns, stall_cta);
}
