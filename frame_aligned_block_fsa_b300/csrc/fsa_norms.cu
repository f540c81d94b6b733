// fsa_norms.cu -- the precomputed norm arrays of the norm-bound softmax.
//
// "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU" (aihot.vn), section
// "Giai phong Softmax": by Cauchy-Schwarz a query's largest logit is at most its norm times
// the largest key norm; a small array of precomputed norms lets each row fix its bound when
// it starts.  The bound is taken over each row's own key set (the window frames and the
// reference frame), which is what makes it valid for the windowed mask.
//
// Three HBM-bound kernels (bf16 rows read with 128-bit loads, 16 threads per 256-byte row):
//   1. key_frame_stats   one block per (frame, head): max key norm of the frame and the
//                        per-frame column sums of K (for the mean key of a key set);
//   2. query_bounds      per (row chunk, frame, head): ||q||, bound = c ||q|| Kmax_S, and the
//                        gap bound c (||q|| Kmax_S - <q, kbar_S>), max-reduced per head;
//   3. eligibility       per head: max gap bound <= tau.
// All reductions run in a fixed order, so the results are deterministic.
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa_internal.h"

namespace fsa {

__device__ __forceinline__ uint4 ldg_stream(const uint4* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4& u, float* x)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Sum over the TPR consecutive lanes that share a row.
template <int TPR>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
__global__ void __launch_bounds__(256) key_frame_stats_kernel(const uint16_t* __restrict__ k, int N, int T,
                                                              int F, float* __restrict__ kmax,
                                                              float* __restrict__ ksum,
                                                              unsigned* __restrict__ gmax)
{
    constexpr int TPR = D / 8;       // threads per row, 16 bytes each
    constexpr int RPI = 256 / TPR;   // rows per block iteration
    __shared__ float cs[RPI][D + 1];
    __shared__ float wmax[8];
    const int g = blockIdx.x, h = blockIdx.y;
    const int sub = threadIdx.x % TPR, rsel = threadIdx.x / TPR;
    const uint4* base = reinterpret_cast<const uint4*>(k + (static_cast<int64_t>(h) * N + static_cast<int64_t>(g) * T) * D);
    float csum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float mx = 0.0f;
    // the trip count is uniform across the block so the row-group shuffles stay converged
#pragma unroll 4
    for (int rb = 0; rb < T; rb += RPI) {
        const int r = rb + rsel;
        float x[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (r < T) unpack8(ldg_stream(base + static_cast<int64_t>(r) * TPR + sub), x);
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ss = fmaf(x[e], x[e], ss);
            csum[e] += x[e];
        }
        ss = group_sum<TPR>(ss);
        mx = fmaxf(mx, sqrtf(ss));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
#pragma unroll
    for (int e = 0; e < 8; ++e) cs[rsel][sub * 8 + e] = csum[e];
    __syncthreads();
    if (threadIdx.x < D) {
        float s = 0.0f;
        for (int r = 0; r < RPI; ++r) s += cs[r][threadIdx.x];
        ksum[(static_cast<int64_t>(h) * F + g) * D + threadIdx.x] = s;
    }
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
        kmax[static_cast<int64_t>(h) * F + g] = m;
        if (g == 0) gmax[h] = 0u;
    }
}

template <int D>
__global__ void __launch_bounds__(256) query_bounds_kernel(
    const uint16_t* __restrict__ q, int N, int T, int F, const int32_t* __restrict__ runs, float scale,
    const float* __restrict__ kmax, const float* __restrict__ ksum, float* __restrict__ qnorm,
    float* __restrict__ bound, unsigned* __restrict__ gmax, int rows_per_block)
{
    constexpr int TPR = D / 8;
    constexpr int RPI = 256 / TPR;
    __shared__ float kbar[D];
    __shared__ float kh_s;
    __shared__ float wmax[8];
    const int f = blockIdx.y, h = blockIdx.z;
    const int32_t* rr = runs + f * kRunStride;
    const int n_runs = rr[0];
    if (threadIdx.x < D) {
        float s = 0.0f;
        int count = 0;
        for (int r = 0; r < n_runs; ++r) {
            const int g0 = rr[1 + 2 * r] / T, ng = rr[2 + 2 * r] / T;
            for (int g = g0; g < g0 + ng; ++g) s += ksum[(static_cast<int64_t>(h) * F + g) * D + threadIdx.x];
            count += rr[2 + 2 * r];
        }
        kbar[threadIdx.x] = s / static_cast<float>(count);
    }
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int r = 0; r < n_runs; ++r) {
            const int g0 = rr[1 + 2 * r] / T, ng = rr[2 + 2 * r] / T;
            for (int g = g0; g < g0 + ng; ++g) m = fmaxf(m, kmax[static_cast<int64_t>(h) * F + g]);
        }
        kh_s = m;
    }
    __syncthreads();
    const float K = kh_s;
    const int sub = threadIdx.x % TPR, rsel = threadIdx.x / TPR;
    float kb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) kb[e] = kbar[sub * 8 + e];
    const int r0 = blockIdx.x * rows_per_block;
    const int r1 = min(T, r0 + rows_per_block);
    const int64_t row_base = static_cast<int64_t>(h) * N + static_cast<int64_t>(f) * T;
    const uint4* base = reinterpret_cast<const uint4*>(q + row_base * D);
    float gworst = 0.0f;
#pragma unroll 4
    for (int rb = r0; rb < r1; rb += RPI) {
        const int r = rb + rsel;
        const bool act = r < r1;
        float x[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (act) unpack8(ldg_stream(base + static_cast<int64_t>(r) * TPR + sub), x);
        float ss = 0.0f, dot = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ss = fmaf(x[e], x[e], ss);
            dot = fmaf(x[e], kb[e], dot);
        }
        ss = group_sum<TPR>(ss);
        dot = group_sum<TPR>(dot);
        const float qn = sqrtf(ss);
        const float qk = qn * K;
        if (act) gworst = fmaxf(gworst, scale * (qk - dot));
        if (act && sub == 0) {
            if (qnorm) qnorm[row_base + r] = qn;
            bound[row_base + r] = scale * qk;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gworst = fmaxf(gworst, __shfl_xor_sync(0xffffffffu, gworst, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = gworst;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
        // non-negative floats order like their bit patterns
        atomicMax(gmax + h, __float_as_uint(fmaxf(m, 0.0f)));
    }
}

__global__ void eligibility_kernel(const unsigned* __restrict__ gmax, float tau, uint8_t* __restrict__ eligible,
                                   int H)
{
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h < H) eligible[h] = static_cast<uint8_t>(__uint_as_float(gmax[h]) <= tau);
}

template <int D>
static int launch_norms_d(const NormsLaunch& L)
{
    key_frame_stats_kernel<D><<<dim3(L.F, L.H), 256, 0, L.stream>>>(L.k, L.N, L.T, L.F, L.kmax, L.ksum, L.gmax);
    const int rows_per_block = 128;
    const dim3 grid((L.T + rows_per_block - 1) / rows_per_block, L.F, L.H);
    query_bounds_kernel<D><<<grid, 256, 0, L.stream>>>(L.q, L.N, L.T, L.F, L.runs, L.scale, L.kmax, L.ksum,
                                                       L.qnorm, L.bound, L.gmax, rows_per_block);
    eligibility_kernel<<<(L.H + 127) / 128, 128, 0, L.stream>>>(L.gmax, L.tau, L.eligible, L.H);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_norms(const NormsLaunch& L)
{
    if (L.D == 64) return launch_norms_d<64>(L);
    if (L.D == 128) return launch_norms_d<128>(L);
    return -2;
}

}  // namespace fsa
