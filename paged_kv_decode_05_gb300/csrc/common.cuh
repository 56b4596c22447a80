// Device helpers shared by the libpkv kernels: element traits, conversions
// and thin inline-PTX wrappers for mbarriers and bulk (TMA) copies.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;      // tokens per physical block
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- traits ---
struct F16 {};
struct BF16 {};
struct I8 {};

template <typename T> struct Elem;
template <> struct Elem<F16>  { static constexpr int bytes = 2; };
template <> struct Elem<BF16> { static constexpr int bytes = 2; };
template <> struct Elem<I8>   { static constexpr int bytes = 1; };

// ------------------------------------------------------------ conversion ---
// Two packed 16-bit values (low half first) -> float2, exact.
__device__ __forceinline__ float2 unpack2(BF16, uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float2 unpack2(F16, uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}
// Two int8 codes c (selected bytes of a word already XOR-ed with 0x80808080,
// i.e. c + 128) -> fp16x2 holding 1152 + c exactly: the byte becomes the low
// mantissa byte of 1024 (fp16 0x6400). The caller removes the 1152 bias.
// `sel` picks the bytes: 0x4140 -> bytes 0,1; 0x4342 -> bytes 2,3.
__device__ __forceinline__ uint32_t i8x2_biased_h2(uint32_t biased, uint32_t sel) {
    return __byte_perm(biased, 0x64646464u, sel);
}

// d += a * b on the tensor cores: m16n8k16, fp16 inputs, fp32 accumulators
// (a: 4 registers of the row-major 16x16 tile, b: 2 of the 16x8 tile).
__device__ __forceinline__ void mma_16816_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += a * b on the tensor cores: m16n8k16 with bf16 or fp16 inputs (the
// cache type; A and B always share it), fp32 accumulators.
template <typename KV>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    if constexpr (std::is_same<KV, BF16>::value)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two floats -> one packed 16-bit pair of the cache type (lo in the low half), RN.
template <typename KV>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (std::is_same<KV, BF16>::value) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

__device__ __forceinline__ float load_scalar(BF16, const void* p, long i) {
    return __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(p)[i]) << 16);
}
__device__ __forceinline__ float load_scalar(F16, const void* p, long i) {
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
}
__device__ __forceinline__ void store_scalar(BF16, void* p, long i, float x) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
}
__device__ __forceinline__ void store_scalar(F16, void* p, long i, float x) {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);
}

// 2^x via the SFU (ex2.approx: relative error ~2^-22; ex2(-inf) = +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ INT8 codes ---
// New code of value x under scale s: clamp(rne(x / s), -127, 127) with an
// IEEE divide; 0 when s == 0.
__device__ __forceinline__ int quant_code(float x, float s) {
    if (s == 0.f) return 0;
    const int q = __float2int_rn(__fdiv_rn(x, s));  // IEEE divide, ties-to-even
    return max(-127, min(127, q));
}
// Four stored codes re-expressed under a grown scale: rne((q * s_o) / s),
// multiply then divide, each IEEE-rounded in fp32.
__device__ __forceinline__ uint32_t requant_word(uint32_t in, float s_o, float s) {
    uint32_t out = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int q = int(int8_t(in >> (8 * b)));
        const float r = __fdiv_rn(__fmul_rn(float(q), s_o), s);
        out |= (uint32_t(__float2int_rn(r)) & 0xffu) << (8 * b);
    }
    return out;
}

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// As mbar_try_wait, but the thread may sleep in the barrier (suspend-time hint
// of 1 ms) until the phase completes, leaving the issue slots to other warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
    return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// of the global timer or 2^26 polls, whichever comes first (the poll cap
// bounds the wait even if the timer were not to advance). Between polls the
// thread sleeps in the barrier.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; !mbar_try_wait_sleep(bar, parity); ++it) {
        if (it >= (1u << 26)) return false;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Order this thread's generic-proxy writes to shared memory before later
// asynchronous-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ bulk copy ---
// One contiguous global -> shared copy by the TMA unit; completion is
// signalled as transaction bytes on `bar`. dst, src 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// 2-D tiled TMA load of box (x, y) of `tmap` into shared memory at `dst`,
// completion signalled as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tmap, int x, int y,
                                            uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}
// 4-byte asynchronous global -> shared copy, tracked by cp.async groups.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (a no-op when launched without
// the attribute), and let the next grid on the stream start launching.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` on `stream` allowing it to overlap the tail of the previous
// grid on the stream; the kernel must call griddep_wait() before it reads
// anything an earlier grid may write.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void flag_status(uint32_t* st, uint32_t bits) {
    if (st) atomicOr(st, bits);
}

}  // namespace pkv
