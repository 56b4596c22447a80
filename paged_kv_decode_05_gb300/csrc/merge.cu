// Merge of partial attention states: the split-K reduce on its own.
//
// Attention over a set of tokens may be computed piece by piece; piece i
// leaves (m_i, l_i, o_i) with m_i its largest score, l_i = sum exp(s - m_i)
// and o_i = sum exp(s - m_i) v (unnormalised). The attention over the union
// is sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i with M = max_i m_i, for
// any partition of the tokens (the flash-decoding reduce that the paged
// decode kernel's combine phase applies to its own pieces; here the caller
// brings the states, e.g. one sequence's pieces gathered from several GPUs).
//
// One warp per (row, head): lanes own float4 columns of the head's D values
// and fold the row's states in order with an online merge (the running sums
// are rescaled whenever the maximum grows), all in fp32; the exponentials are
// taken in base 2 of the differences scaled by log2 e.
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMaxHeadDim = 512;
constexpr float kLog2eM = 1.4426950408889634f;

struct MergeParams {
    const float* m;        // [S, H]
    const float* l;        // [S, H]
    const float4* o;       // [S, H, D/4]
    const int32_t* row_ptr;
    void* out;             // [R, H, D] out dtype
    float* out_m;          // [R, H] or nullptr
    float* out_l;
    uint32_t* status;
    long long num_states;
    int rows, heads, d4;
};

template <typename QT>
__device__ __forceinline__ void store4(void* out, long long i4, float4 v, float s) {
    uint2 w;
    if constexpr (std::is_same<QT, BF16>::value) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x * s, v.y * s);
        __nv_bfloat162 b = __floats2bfloat162_rn(v.z * s, v.w * s);
        w = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    } else {
        __half2 a = __floats2half2_rn(v.x * s, v.y * s);
        __half2 b = __floats2half2_rn(v.z * s, v.w * s);
        w = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    reinterpret_cast<uint2*>(out)[i4] = w;
}

template <typename QT, int NV>
__global__ void __launch_bounds__(kMergeThreads) merge_states_kernel(const MergeParams p) {
    griddep_wait();
    const long long item = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (item >= (long long)p.rows * p.heads) return;
    const long long r = item / p.heads;
    const int h = int(item - r * p.heads);
    long long s0 = p.row_ptr[r], s1 = p.row_ptr[r + 1];
    if (s0 < 0 || s1 < s0 || s1 > p.num_states) {   // bad range: flagged, row left as zeros
        if (lane == 0) flag_status(p.status, PKV_DEV_BAD_INDEX);
        s0 = s1 = 0;
    }
    float M = -INFINITY, den = 0.f;                  // running max of m (natural units)
    float4 num[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) num[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long s = s0; s < s1; ++s) {
        const long long sh = s * p.heads + h;
        const float ms = __ldg(p.m + sh), ls = __ldg(p.l + sh);
        if (!(ms > -INFINITY) || !(ls > 0.f)) continue;   // empty piece (or NaN m)
        if (ms > M) {
            const float a = (M == -INFINITY) ? 0.f : fast_exp2((M - ms) * kLog2eM);
            den *= a;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                num[k].x *= a; num[k].y *= a; num[k].z *= a; num[k].w *= a;
            }
            M = ms;
        }
        const float a = fast_exp2((ms - M) * kLog2eM);
        den = fmaf(a, ls, den);
        const float4* os = p.o + sh * p.d4;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = lane + 32 * k;
            if (c < p.d4) {
                const float4 v = __ldg(os + c);
                num[k].x = fmaf(a, v.x, num[k].x); num[k].y = fmaf(a, v.y, num[k].y);
                num[k].z = fmaf(a, v.z, num[k].z); num[k].w = fmaf(a, v.w, num[k].w);
            }
        }
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = lane + 32 * k;
        if (c < p.d4) store4<QT>(p.out, item * p.d4 + c, num[k], inv);
    }
    if (lane == 0) {
        if (p.out_m) p.out_m[item] = M;
        if (p.out_l) p.out_l[item] = den;
    }
    griddep_launch_dependents();
}

template <typename QT>
cudaError_t launch_merge(const MergeParams& p, int grid, cudaStream_t st) {
    const int nv = (p.d4 + 31) / 32;
    if (nv <= 1) return launch_pdl(merge_states_kernel<QT, 1>, dim3(grid), dim3(kMergeThreads), 0, st, p);
    if (nv <= 2) return launch_pdl(merge_states_kernel<QT, 2>, dim3(grid), dim3(kMergeThreads), 0, st, p);
    return launch_pdl(merge_states_kernel<QT, 4>, dim3(grid), dim3(kMergeThreads), 0, st, p);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace pkv

// ------------------------------------------------------------------- host ---
using namespace pkv;

extern "C" pkv_status pkv_merge_states(const float* part_m, const float* part_l,
                                       const float* part_o, int64_t num_states,
                                       const int32_t* row_ptr, int32_t num_rows,
                                       int32_t num_heads, int32_t head_dim, pkv_dtype out_dtype,
                                       void* out, float* out_m, float* out_l,
                                       uint32_t* dev_status, cudaStream_t stream) {
    if (num_rows < 0 || num_heads <= 0 || num_states < 0) return PKV_ERR_INVALID_ARG;
    if (head_dim <= 0 || head_dim % 4 != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim > kMaxHeadDim) return PKV_ERR_UNSUPPORTED;
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (num_rows == 0) return PKV_OK;
    if (!row_ptr || !out || !aligned_to(row_ptr, 4) || !aligned_to(out, 8)) return PKV_ERR_INVALID_ARG;
    if (num_states > 0 && (!part_m || !part_l || !part_o || !aligned_to(part_m, 4) ||
                           !aligned_to(part_l, 4) || !aligned_to(part_o, 16)))
        return PKV_ERR_INVALID_ARG;
    if ((out_m && !aligned_to(out_m, 4)) || (out_l && !aligned_to(out_l, 4)) ||
        (dev_status && !aligned_to(dev_status, 4)))
        return PKV_ERR_INVALID_ARG;
    const long long items = (long long)num_rows * num_heads;
    const long long grid = (items + kMergeWarps - 1) / kMergeWarps;
    if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    MergeParams p;
    p.m = part_m; p.l = part_l; p.o = reinterpret_cast<const float4*>(part_o);
    p.row_ptr = row_ptr; p.out = out; p.out_m = out_m; p.out_l = out_l;
    p.status = dev_status; p.num_states = num_states;
    p.rows = num_rows; p.heads = num_heads; p.d4 = head_dim / 4;
    const cudaError_t e = out_dtype == PKV_BF16 ? launch_merge<BF16>(p, int(grid), stream)
                                                 : launch_merge<F16>(p, int(grid), stream);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}
