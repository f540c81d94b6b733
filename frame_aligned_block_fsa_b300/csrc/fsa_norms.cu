// fsa_norms.cu -- the precomputed norm arrays of the norm-bound softmax.
//
// "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU" (aihot.vn), section
// "Giai phong Softmax": by Cauchy-Schwarz a query's largest logit is at most its norm times
// the largest key norm; a small array of precomputed norms lets each row fix its bound when
// it starts.  The bound is taken over each row's own key set (the window frames and the
// reference frame), which is what makes it valid for the windowed mask.
//
// Three HBM-bound kernels (bf16 rows read with 128-bit loads, D/16 threads per row, packed
// f32x2 arithmetic):
//   1. key_frame_stats   per (chunk of a frame's rows, frame, head): the chunk's max key norm
//                        and column sums of K; the last chunk of a frame to finish reduces
//                        the chunks in a fixed order into the frame's max key norm and key
//                        sums (a ticket counter, no waiting);
//   2. query_bounds      per (row chunk, frame, head): ||q||, bound = c ||q|| Kmax_S, and the
//                        gap bound c (||q|| Kmax_S - <q, kbar_S>), max-reduced per head; the
//                        last block of a head to finish (a ticket counter) sets its
//                        eligibility: max gap bound <= tau.
// The query pass is a programmatic dependent launch: its blocks start while the key pass's last
// blocks run, issue their first query loads, and wait for the key pass (griddepcontrol.wait)
// only before they read its statistics.
// With mean-centred keys (same section: keys share a large common component; subtracting
// their mean tightens the bound and the softmax does not see it) the last frame of a head to
// finish also forms the head's key mean mu from the frame sums, a second pass over K
// (key_centred_max) takes max ||k - mu|| per frame, and query_bounds uses
// c (||q|| Kmax_S + <q, mu>): Cauchy-Schwarz on the centred logit with the row constant
// c <q, mu> added back, so it bounds the uncentred logits and the lse needs no correction.
// All reductions run in a fixed order (or take a max), so the results are deterministic.
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

constexpr int kNormThreads = 256;

// Programmatic dependent launch: a kernel lets the next one in the stream start (its blocks
// may become resident once every block of this one has run this), and the next one waits for
// this one to complete, with its writes visible, before it reads them.
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
constexpr int kBatch = 2;  // row iterations whose loads are issued together (2 x 2 x 16 B per thread)

// A thread reads 16 bf16 of a row as two 16-byte loads, D/2 columns apart, so that the row's
// D/16 threads cover a contiguous half-row with each load.  Its columns are
// [8 sub, 8 sub + 8) and [D/2 + 8 sub, D/2 + 8 sub + 8).
template <int D>
__device__ __forceinline__ void load_row16(const uint4* row, int sub, bool act, uint4& a, uint4& b)
{
    if (act) {
        a = ldg_stream(row + sub);
        b = ldg_stream(row + D / 16 + sub);
    } else {
        a = make_uint4(0u, 0u, 0u, 0u);
        b = a;
    }
}

// The 16 values of a thread as 8 pairs (x[2i], x[2i+1]).
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float2* x)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <int D>
__global__ void __launch_bounds__(kNormThreads) key_frame_stats_kernel(
    const uint16_t* __restrict__ k, int N, int T, int F, int chunks, int rows_per_chunk,
    float* __restrict__ part_max, float* __restrict__ part_sum, unsigned* __restrict__ tickets,
    float* __restrict__ kmax, float* __restrict__ ksum, unsigned* __restrict__ gmax, int center,
    float* __restrict__ mu, unsigned* __restrict__ htickets)
{
    constexpr int TPR = D / 16;                // threads per row, 16 values each
    constexpr int RPI = kNormThreads / TPR;    // rows per block iteration
    __shared__ float cs[RPI][D + 1];
    __shared__ float wmax[kNormThreads / 32];
    __shared__ bool last;
    const int c = blockIdx.x, g = blockIdx.y, h = blockIdx.z;
    pdl_allow_dependents();
    const int sub = threadIdx.x % TPR, rsel = threadIdx.x / TPR;
    const int r0 = c * rows_per_chunk;
    const int r1 = min(T, r0 + rows_per_chunk);
    const uint4* base = reinterpret_cast<const uint4*>(k + (static_cast<int64_t>(h) * N + static_cast<int64_t>(g) * T) * D);
    float2 csum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) csum[i] = make_float2(0.0f, 0.0f);
    float mx = 0.0f;
    // the trip count is uniform across the block so the row-group shuffles stay converged
    for (int rb = r0; rb < r1; rb += kBatch * RPI) {
        uint4 ua[kBatch], ub[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = rb + b * RPI + rsel;
            load_row16<D>(base + static_cast<int64_t>(r) * (D / 8), sub, r < r1, ua[b], ub[b]);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            float2 x[8];
            unpack16(ua[b], ub[b], x);
            float2 ss = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ss = fma2(x[i], x[i], ss);
                csum[i] = add2(csum[i], x[i]);
            }
            const float n2 = group_sum<TPR>(ss.x + ss.y);
            mx = fmaxf(mx, sqrtf(n2));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // pair i holds columns (2i, 2i+1) of the thread's 16: the first 4 pairs lie in the
        // first half-row, the last 4 in the second
        const int col = (i < 4 ? 8 * sub + 2 * i : D / 2 + 8 * sub + 2 * (i - 4));
        cs[rsel][col] = csum[i].x;
        cs[rsel][col + 1] = csum[i].y;
    }
    __syncthreads();
    const int64_t hg = static_cast<int64_t>(h) * F + g;
    if (threadIdx.x < D) {
        float s = 0.0f;
        for (int r = 0; r < RPI; ++r) s += cs[r][threadIdx.x];
        part_sum[(hg * chunks + c) * D + threadIdx.x] = s;
    }
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int w = 1; w < kNormThreads / 32; ++w) m = fmaxf(m, wmax[w]);
        part_max[hg * chunks + c] = m;
        if (c == 0 && g == 0) gmax[h] = 0u;
    }
    // The last chunk of this frame to finish reduces all chunks, in chunk order.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(tickets + hg, 1u);
        last = ticket == static_cast<unsigned>(chunks - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (threadIdx.x < D) {
        float s = 0.0f;
        for (int i = 0; i < chunks; ++i) s += __ldcg(part_sum + (hg * chunks + i) * D + threadIdx.x);
        ksum[hg * D + threadIdx.x] = s;
    }
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int i = 0; i < chunks; ++i) m = fmaxf(m, __ldcg(part_max + hg * chunks + i));
        // centred: zero here, max-reduced by key_centred_max in the next launch
        kmax[hg] = center ? 0.0f : m;
        tickets[hg] = 0u;  // ready for the next launch
    }
    if (!center) return;
    // The last frame of this head to finish forms the head's key mean, in frame order.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(htickets + h, 1u);
        last = ticket == static_cast<unsigned>(F - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (threadIdx.x < D) {
        float s = 0.0f;
        for (int gg = 0; gg < F; ++gg) s += __ldcg(ksum + (static_cast<int64_t>(h) * F + gg) * D + threadIdx.x);
        mu[static_cast<int64_t>(h) * D + threadIdx.x] = s / static_cast<float>(N);
    }
    if (threadIdx.x == 0) htickets[h] = 0u;
}

// Max over a chunk of a frame's keys of ||k - mu_h||, max-reduced into kmax[h][g] (zeroed by
// key_frame_stats; non-negative floats order like their bit patterns).
template <int D>
__global__ void __launch_bounds__(kNormThreads) key_centred_max_kernel(
    const uint16_t* __restrict__ k, int N, int T, int F, int rows_per_chunk, const float* __restrict__ mu,
    float* __restrict__ kmax)
{
    constexpr int TPR = D / 16;
    constexpr int RPI = kNormThreads / TPR;
    __shared__ float wmax[kNormThreads / 32];
    const int c = blockIdx.x, g = blockIdx.y, h = blockIdx.z;
    pdl_allow_dependents();
    const int sub = threadIdx.x % TPR, rsel = threadIdx.x / TPR;
    const int r0 = c * rows_per_chunk;
    const int r1 = min(T, r0 + rows_per_chunk);
    const uint4* base = reinterpret_cast<const uint4*>(k + (static_cast<int64_t>(h) * N + static_cast<int64_t>(g) * T) * D);
    float2 nmu[8];  // minus the mean, at this thread's 16 columns
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int col = (i < 4 ? 8 * sub + 2 * i : D / 2 + 8 * sub + 2 * (i - 4));
        nmu[i] = make_float2(-mu[static_cast<int64_t>(h) * D + col], -mu[static_cast<int64_t>(h) * D + col + 1]);
    }
    float mx = 0.0f;
    for (int rb = r0; rb < r1; rb += kBatch * RPI) {
        uint4 ua[kBatch], ub[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = rb + b * RPI + rsel;
            load_row16<D>(base + static_cast<int64_t>(r) * (D / 8), sub, r < r1, ua[b], ub[b]);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const bool act = rb + b * RPI + rsel < r1;
            float2 x[8];
            unpack16(ua[b], ub[b], x);
            float2 ss = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 d = add2(x[i], nmu[i]);
                ss = fma2(d, d, ss);
            }
            const float n2 = group_sum<TPR>(ss.x + ss.y);
            // an inactive row reads zeros, whose distance to the mean is no key's
            if (act) mx = fmaxf(mx, sqrtf(n2));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int w = 1; w < kNormThreads / 32; ++w) m = fmaxf(m, wmax[w]);
        atomicMax(reinterpret_cast<unsigned*>(kmax) + static_cast<int64_t>(h) * F + g, __float_as_uint(m));
    }
}

template <int D, bool CENTER>
__global__ void __launch_bounds__(kNormThreads) query_bounds_kernel(
    const uint16_t* __restrict__ q, int N, int T, int F, const int32_t* __restrict__ runs, float scale,
    const float* __restrict__ kmax, const float* __restrict__ ksum, const float* __restrict__ mu,
    float* __restrict__ qnorm, float* __restrict__ bound, unsigned* __restrict__ gmax, int rows_per_block,
    float tau, uint8_t* __restrict__ eligible, unsigned* __restrict__ etickets, int blocks_per_head)
{
    constexpr int TPR = D / 16;
    constexpr int RPI = kNormThreads / TPR;
    __shared__ float kbar[D];
    __shared__ float kh_s;
    __shared__ float wmax[kNormThreads / 32];
    __shared__ bool last;
    const int f = blockIdx.y, h = blockIdx.z;
    const int sub = threadIdx.x % TPR, rsel = threadIdx.x / TPR;
    const int r0 = blockIdx.x * rows_per_block;
    const int r1 = min(T, r0 + rows_per_block);
    const int64_t row_base = static_cast<int64_t>(h) * N + static_cast<int64_t>(f) * T;
    const uint4* base = reinterpret_cast<const uint4*>(q + row_base * D);
    // The first batch of query rows is in flight while the key statistics of the row's key
    // set are gathered from L2.
    uint4 ua[kBatch], ub[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
        const int r = r0 + b * RPI + rsel;
        load_row16<D>(base + static_cast<int64_t>(r) * (D / 8), sub, r < r1, ua[b], ub[b]);
    }
    // the key statistics (and the zeroed gap maximum) come from the key pass
    pdl_wait_prerequisite();
    const int32_t* rr = runs + f * kRunStride;
    const int n_runs = rr[0];
    if (threadIdx.x < D) {
        float s = 0.0f;
        int count = 0;
        for (int r = 0; r < n_runs; ++r) {
            const int g0 = rr[1 + 2 * r] / T, ng = rr[2 + 2 * r] / T;
            const float* src = ksum + (static_cast<int64_t>(h) * F + g0) * D + threadIdx.x;
#pragma unroll 8
            for (int g = 0; g < ng; ++g) s += src[static_cast<int64_t>(g) * D];
            count += rr[2 + 2 * r];
        }
        kbar[threadIdx.x] = s / static_cast<float>(count);
    } else if (threadIdx.x < D + 32) {
        // one warp: the largest key norm of the key set, one frame per lane
        const int lane = threadIdx.x - D;
        float m = 0.0f;
        for (int r = 0; r < n_runs; ++r) {
            const int g0 = rr[1 + 2 * r] / T, ng = rr[2 + 2 * r] / T;
            for (int i = lane; i < ng; i += 32) m = fmaxf(m, kmax[static_cast<int64_t>(h) * F + g0 + i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) kh_s = m;
    }
    __syncthreads();
    const float K = kh_s;
    float2 kb[8], mb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int col = (i < 4 ? 8 * sub + 2 * i : D / 2 + 8 * sub + 2 * (i - 4));
        kb[i] = make_float2(kbar[col], kbar[col + 1]);
        if (CENTER) mb[i] = make_float2(mu[static_cast<int64_t>(h) * D + col], mu[static_cast<int64_t>(h) * D + col + 1]);
    }
    float gworst = 0.0f;
    for (int rb = r0; rb < r1; rb += kBatch * RPI) {
        if (rb != r0) {
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int r = rb + b * RPI + rsel;
                load_row16<D>(base + static_cast<int64_t>(r) * (D / 8), sub, r < r1, ua[b], ub[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = rb + b * RPI + rsel;
            const bool act = r < r1;
            float2 x[8];
            unpack16(ua[b], ub[b], x);
            float2 ss = make_float2(0.0f, 0.0f), dot = make_float2(0.0f, 0.0f), qm = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ss = fma2(x[i], x[i], ss);
                dot = fma2(x[i], kb[i], dot);
                if (CENTER) qm = fma2(x[i], mb[i], qm);
            }
            const float n2 = group_sum<TPR>(ss.x + ss.y);
            const float dt = group_sum<TPR>(dot.x + dot.y);
            const float qn = sqrtf(n2);
            // the bound before the factor c: ||q|| Kmax_S, centred ||q|| Kmax_S + <q, mu>
            const float qk = CENTER ? fmaf(qn, K, group_sum<TPR>(qm.x + qm.y)) : qn * K;
            if (act) gworst = fmaxf(gworst, scale * (qk - dt));
            if (act && sub == 0) {
                if (qnorm) qnorm[row_base + r] = qn;
                bound[row_base + r] = scale * qk;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gworst = fmaxf(gworst, __shfl_xor_sync(0xffffffffu, gworst, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = gworst;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int w = 1; w < kNormThreads / 32; ++w) m = fmaxf(m, wmax[w]);
        // non-negative floats order like their bit patterns
        atomicMax(gmax + h, __float_as_uint(fmaxf(m, 0.0f)));
        // the last block of this head to finish sets the head's eligibility
        __threadfence();
        last = atomicAdd(etickets + h, 1u) == static_cast<unsigned>(blocks_per_head - 1);
    }
    __syncthreads();
    if (last && threadIdx.x == 0) {
        __threadfence();
        eligible[h] = static_cast<uint8_t>(__uint_as_float(__ldcg(gmax + h)) <= tau);
        etickets[h] = 0u;  // ready for the next launch
    }
}

__global__ void eligibility_kernel(const unsigned* __restrict__ gmax, float tau, uint8_t* __restrict__ eligible,
                                   int H)
{
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h < H) eligible[h] = static_cast<uint8_t>(__uint_as_float(gmax[h]) <= tau);
}

int norms_key_chunks(int T)
{
    const int c = T / 256;  // about 256-300 rows per block at the workload sizes
    return c < 1 ? 1 : (c > kMaxKeyChunks ? kMaxKeyChunks : c);
}

template <int D>
static int launch_norms_d(const NormsLaunch& L)
{
    const int chunks = norms_key_chunks(L.T);
    const int rows_per_chunk = (L.T + chunks - 1) / chunks;
    key_frame_stats_kernel<D><<<dim3(chunks, L.F, L.H), kNormThreads, 0, L.stream>>>(
        L.k, L.N, L.T, L.F, chunks, rows_per_chunk, L.part_max, L.part_sum, L.tickets, L.kmax, L.ksum, L.gmax,
        L.center, L.mu, L.htickets);
    if (L.center)
        key_centred_max_kernel<D><<<dim3(chunks, L.F, L.H), kNormThreads, 0, L.stream>>>(L.k, L.N, L.T, L.F,
                                                                                         rows_per_chunk, L.mu, L.kmax);
    // about 256 query rows per block, split evenly over a frame (T = 1200: 5 blocks of 240)
    const int qblocks = (L.T + 255) / 256;
    const int rows_per_block = (L.T + qblocks - 1) / qblocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(qblocks, L.F, L.H);
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    unsigned* etickets = L.htickets + L.H;
    const cudaError_t e =
        L.center ? cudaLaunchKernelEx(&cfg, query_bounds_kernel<D, true>, L.q, L.N, L.T, L.F, L.runs, L.scale,
                                      static_cast<const float*>(L.kmax), static_cast<const float*>(L.ksum),
                                      static_cast<const float*>(L.mu), L.qnorm, L.bound, L.gmax, rows_per_block,
                                      L.tau, L.eligible, etickets, qblocks * L.F)
                 : cudaLaunchKernelEx(&cfg, query_bounds_kernel<D, false>, L.q, L.N, L.T, L.F, L.runs, L.scale,
                                      static_cast<const float*>(L.kmax), static_cast<const float*>(L.ksum),
                                      static_cast<const float*>(nullptr), L.qnorm, L.bound, L.gmax, rows_per_block,
                                      L.tau, L.eligible, etickets, qblocks * L.F);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return -3;
    }
    return launch_status();
}

int launch_eligibility(const unsigned* gmax, float tau, uint8_t* eligible, int H, cudaStream_t stream)
{
    eligibility_kernel<<<(H + 127) / 128, 128, 0, stream>>>(gmax, tau, eligible, H);
    return launch_status();
}

int launch_norms(const NormsLaunch& L)
{
    if (L.D == 64) return launch_norms_d<64>(L);
    if (L.D == 128) return launch_norms_d<128>(L);
    return -2;
}

}  // namespace fsa
