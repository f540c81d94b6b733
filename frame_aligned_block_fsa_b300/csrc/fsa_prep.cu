// fsa_prep.cu -- the attention's inputs prepared in one pass: RMS norm, QKV projection,
// rotary embedding, head packing, and the bound's norms as a by-product.
//
// "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU" (aihot.vn), section
// "Bo cuc la ABI", Fig. 5: the chain of small operations that produces the attention's inputs
// (normalisation, rotary embeddings, projection, head packing) is fused into one kernel that
// writes its output in exactly the layout the next step reads, so no repacking copies are
// left between them.  Here the next step is the attention kernel: the projection's epilogue
// writes Q, K and V as bf16 [H][N][D] (the layout of its TMA tensor maps) and, while the
// values are in registers, the norms the norm-bound softmax needs (section "Giai phong
// Softmax"), so no separate pass re-reads Q and K for them.
//
// Readings (the pages name the steps, not their exact form): RMS norm without a learned gain
// (a gain folds into the weights); y = xhat W^T with W bf16 [3 H D][d_model] (q rows, then k,
// then v, head-major); rotary embedding of q and k at position = token index, pairs
// (i, i + D/2) turned by n * base^(-2i/D); v not rotated.
//
// Kernels, in stream order:
//   rms_kernel          1 / rms of every token row (one warp per row)
//   fsa_prep_kernel     the projection GEMM, one cooperative launch, tiles of the K and V
//                       columns first, then of the Q columns.  K/V tile epilogues: rotary, bf16
//                       rounding, the head-packed store, per-frame max key norms (an atomic
//                       max) and per-32-row column sums of K (fixed-order partials).  Before its
//                       first Q epilogue every CTA meets the others at a grid barrier; then the
//                       CTAs share out the per-frame key sums and, after a second barrier, the
//                       max key norm and mean key of every query frame's key set (fixed orders
//                       throughout), and meet a third time.  Q tile epilogues: rotary, rounding,
//                       store, and per row ||q||, the bound c ||q|| Kmax_S and the gap statistic
//                       c (||q|| Kmax_S - <q, kbar_S>), max-reduced per head.  The mainloop of a
//                       CTA's first Q tile runs while its epilogue warps are at the barriers.
//   eligibility         (the norms' kernel) per head: gap maximum <= tau
//
// fsa_prep_kernel (persistent, one CTA per SM, 10 warps): a 256 x 256 output tile is two
// M = 128 accumulators (token rows 0-127 and 128-255) of 256 fp32 TMEM columns each, built by
// tcgen05.mma (kind::f16, bf16 inputs from 128-byte swizzled shared memory, K-major A and B)
// over 64-wide K steps fed by TMA through a 3-stage ring.  The 256 columns are two heads of
// q, k or v (H is even); each of the 8 epilogue warps owns 32 rows (its TMEM lane quarter of
// one accumulator) and takes the two heads in turn: it reads the pairs (i, i + 64) of its rows
// from TMEM, scales by 1/rms, rotates, rounds, and stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa_internal.h"
#include "fsa_ptx.cuh"

namespace fsa {

namespace {

constexpr int kPrepThreads = 320;  // 8 epilogue warps, the TMA warp, the MMA warp
constexpr int kPrepWarpTma = 8, kPrepWarpMma = 9;

struct PrepCfg {
    static constexpr int BM = 256, BN = 256, BK = 64;
    static constexpr int A_BYTES = BM * 128;  // 256 rows x 64 bf16 (one 128-byte swizzle panel)
    static constexpr int B_BYTES = BN * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int NS = 3;
    static constexpr int BAR_OFF = NS * STAGE_BYTES;
    static constexpr int B_FULL = 0;              // NS: A and B of a stage landed
    static constexpr int B_EMPTY = NS;            // NS: the MMAs reading a stage are done
    static constexpr int B_ACC_FULL = 2 * NS;     // the tile's accumulators are complete
    static constexpr int B_ACC_EMPTY = 2 * NS + 1;  // the epilogue has read them (8 arrivals)
    static constexpr int B_DRAIN = 2 * NS + 2;
    static constexpr int N_BARS = 2 * NS + 3;
    static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;  // abort flag +0, TMEM address +8
    static_assert(MISC_OFF + 16 <= BAR_OFF + 256, "reserved area");
    // rotary angles by addition: (cos, sin) of l * theta_i for l < 32 ([i][l], 16 KB) and of
    // n_first * theta_i for each epilogue warp's first row ([warp][i], 4 KB)
    static constexpr int DELTA_OFF = BAR_OFF + 256;
    static constexpr int RBASE_OFF = DELTA_OFF + 64 * 32 * 8;
    static constexpr int SMEM_BYTES = 1024 + RBASE_OFF + 8 * 64 * 8;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, 256, false, false);
};

enum : int { SITE_PREP_EMPTY = 11, SITE_PREP_FULL = 12, SITE_PREP_ACC_EMPTY = 13, SITE_PREP_ACC_FULL = 14,
             SITE_PREP_DRAIN = 15, SITE_PREP_GRID = 16 };

// Output tile t: token-row tile m and 256-column tile nt (K and V tiles first, then Q).  Each
// of the q, k and v sections spans H D / 256 column tiles.
template <int D>
__device__ __forceinline__ void prep_tile(const PrepParams& p, int t, int& m, int& nt)
{
    const int ts = p.H * D / 256;
    if (t < p.tiles_kv) {
        m = t / (2 * ts);
        nt = ts + t % (2 * ts);
    } else {
        const int u = t - p.tiles_kv;
        m = u / ts;
        nt = u % ts;
    }
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// All CTAs' 256 epilogue threads meet here (every CTA of the launch is resident: cooperative
// launch).  Bounded: a wait that gives up raises the CTA's abort flag and records the site.
__device__ __forceinline__ void grid_sync(unsigned* counter, unsigned n, int et, const WaitCtl& wc)
{
    __threadfence();  // this thread's writes (and atomics) are visible device-wide
    __syncwarp();     // the warp is converged for the aligned barrier
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (et == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        const long long t0 = clock64();
        while (ld_acquire_gpu(counter) < n) {
            if (*wc.abort) break;
            if (clock64() - t0 > wc.limit) {
                *wc.abort = 1;
                if (wc.err_word) atomicCAS(wc.err_word, 0, -4 /* FSA_ERR_TIMEOUT */);
                if (wc.err_site) atomicCAS(wc.err_site, 0, SITE_PREP_GRID);
                break;
            }
        }
    }
    __syncwarp();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    __threadfence();
}

// Between the K/V and the Q epilogues: the per-frame key sums from the 32-row partials (added
// in ascending row order, 16 loads in flight), then per query frame f the max key norm and the
// mean key over its key set S(f) (frames in run order), shared out over all CTAs' epilogue
// threads.  Also zeroes the gap maxima before any Q epilogue max-reduces into them.
template <int D>
__device__ void prep_key_stats(const PrepParams& p, int et, const WaitCtl& wc)
{
    const unsigned n = gridDim.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * 256;
    const int64_t total = static_cast<int64_t>(p.H) * p.F * D;
    const int64_t nb32 = (static_cast<int64_t>(p.N) + 31) / 32;
    grid_sync(p.gsync + 0, n, et, wc);  // every K tile's partials and maxima are written
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * 256 + et; e < total; e += stride) {
        const int d = static_cast<int>(e % D);
        const int64_t hg = e / D;
        const int g = static_cast<int>(hg % p.F), h = static_cast<int>(hg / p.F);
        const float* part = p.kpart + static_cast<int64_t>(h) * nb32 * 2 * D;
        const int64_t first = static_cast<int64_t>(g) * p.T, last = first + p.T - 1;
        const int64_t b0 = first / 32, b1 = last / 32;
        float s = 0.0f;
        for (int64_t bb = b0; bb <= b1; bb += 16) {
            float x[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int64_t b = bb + u;
                // a block whose first row lies in an earlier frame holds frame g's rows in side 1
                const int side = b * 32 < first ? 1 : 0;
                x[u] = b <= b1 ? __ldcg(part + (b * 2 + side) * D + d) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (bb + u <= b1) s += x[u];
        }
        p.ksum[e] = s;
    }
    grid_sync(p.gsync + 1, n, et, wc);  // every frame sum is written
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * 256 + et; e < total; e += stride) {
        const int d = static_cast<int>(e % D);
        const int64_t hf = e / D;
        const int f = static_cast<int>(hf % p.F), h = static_cast<int>(hf / p.F);
        const int32_t* rr = p.runs + f * kRunStride;
        float s = 0.0f, m = 0.0f;
        int count = 0;
        for (int r = 0; r < rr[0]; ++r) {
            const int g0 = rr[1 + 2 * r] / p.T, ng = rr[2 + 2 * r] / p.T;
            for (int g = g0; g < g0 + ng; ++g) {
                s += __ldcg(p.ksum + (static_cast<int64_t>(h) * p.F + g) * D + d);
                m = fmaxf(m, __uint_as_float(__ldcg(p.kmax + static_cast<int64_t>(h) * p.F + g)));
            }
            count += rr[2 + 2 * r];
        }
        p.kbar[e] = s / static_cast<float>(count);
        if (d == 0) {
            p.ks[hf] = m;
            if (f == 0) p.gmax[h] = 0u;
        }
    }
    grid_sync(p.gsync + 2, n, et, wc);  // the key-set statistics are written
}

// After the call, lane l holds the sum over the warp's lanes of v[l] (five butterfly rounds,
// each halving the values a lane keeps; the order of the additions is fixed).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool up = lane & 16;
        const float send = up ? v[i] : v[i + 16];
        const float keep = up ? v[i + 16] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 8;
        const float send = up ? v[i] : v[i + 8];
        const float keep = up ? v[i + 8] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 4;
        const float send = up ? v[i] : v[i + 4];
        const float keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 2;
        const float send = up ? v[i] : v[i + 2];
        const float keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    {
        const bool up = lane & 1;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    return v[0];
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 32-byte store (one full sector per lane); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* r)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One epilogue warp: 32 token rows (n_first + lane) of one head of q (sect 0), k (1) or v (2),
// read from TMEM at `trow` (this warp's lane quarter, the head's first column).  The rotary
// angle of row n_first + l and pair i is n_first theta_i + l theta_i: its cosine and sine come
// from rbase[i] (the warp's first row) and delta[i][l] by the addition formulas.
template <int D>
__device__ __forceinline__ void prep_epilogue(const PrepParams& p, uint32_t trow, int sect, int h, int n_first,
                                              int lane, float ri, const float2* delta, const float2* rbase)
{
    constexpr int HALF = D / 2;     // rotary pairs (i, i + D/2)
    constexpr int CHUNKS = D / 32;  // 16 pairs a chunk
    const int n = n_first + lane;
    const bool valid = n < p.N;
    const int nn = valid ? n : p.N - 1;
    const int f = nn / p.T;
    uint16_t* base = sect == 0 ? p.q : (sect == 1 ? p.k : p.v);
    uint4* dst = reinterpret_cast<uint4*>(base + (static_cast<int64_t>(h) * p.N + nn) * D);
    // rows are 2 D bytes, so 32-byte stores need only a 32-byte aligned tensor (uniform test)
    const bool wide = (reinterpret_cast<uintptr_t>(base) & 31u) == 0;
    const float4* kbar = reinterpret_cast<const float4*>(p.kbar + (static_cast<int64_t>(h) * p.F + f) * D);
    // frame segments of the warp's rows (a 32-row block meets at most two frames, T >= 16)
    const int f_lo = n_first / p.T;
    const int n_last = min(n_first + 31, p.N - 1);
    const bool straddle = n_last / p.T != f_lo;
    const int64_t nb32 = (static_cast<int64_t>(p.N) + 31) / 32;
    float* kpart = p.kpart + ((static_cast<int64_t>(h) * nb32 + n_first / 32) * 2) * D;

    float ss = 0.0f, dot = 0.0f;
    // chunk c: pairs 16c .. 16c+15, i.e. columns 16c.. and D/2 + 16c..; the next chunk's TMEM
    // loads are in flight while this one is processed
    float na[16], nb[16];
    tmem_ld_x16(trow, na);
    tmem_ld_x16(trow + HALF, nb);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        float a[16], b[16];
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            reg_fence(na[i]);
            reg_fence(nb[i]);
            a[i] = na[i];
            b[i] = nb[i];
        }
        if (c + 1 < CHUNKS) {
            tmem_ld_x16(trow + 16 * (c + 1), na);
            tmem_ld_x16(trow + HALF + 16 * (c + 1), nb);
        }
        if (sect < 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 cb = rbase[16 * c + i];               // same for every lane: broadcast
                const float2 cd = delta[(16 * c + i) * 32 + lane];  // consecutive lanes: no conflict
                const float cs = cb.x * cd.x - cb.y * cd.y;
                const float sn = cb.y * cd.x + cb.x * cd.y;
                const float x = a[i] * ri, y = b[i] * ri;
                a[i] = x * cs - y * sn;
                b[i] = x * sn + y * cs;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                a[i] *= ri;
                b[i] *= ri;
            }
        }
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            pa[i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
            pb[i] = pack_bf16x2(b[2 * i], b[2 * i + 1]);
        }
        if (valid) {
            if (wide) {
                st_global_v8(dst + 2 * c, pa);
                st_global_v8(dst + HALF / 8 + 2 * c, pb);
            } else {
                dst[2 * c] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                dst[2 * c + 1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
                dst[HALF / 8 + 2 * c] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
                dst[HALF / 8 + 2 * c + 1] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
            }
        }
        if (sect == 2) continue;
        // the norms use the rounded values, the ones the attention kernel will read
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ss = fmaf(bf16_lo(pa[i]), bf16_lo(pa[i]), ss);
            ss = fmaf(bf16_hi(pa[i]), bf16_hi(pa[i]), ss);
            ss = fmaf(bf16_lo(pb[i]), bf16_lo(pb[i]), ss);
            ss = fmaf(bf16_hi(pb[i]), bf16_hi(pb[i]), ss);
        }
        if (sect == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // written earlier in this launch by other CTAs: read from L2, not through L1
                const float4 ka = __ldcg(kbar + 4 * c + i);             // columns 16c + 4i ..
                const float4 kb = __ldcg(kbar + HALF / 4 + 4 * c + i);  // columns D/2 + 16c + 4i ..
                dot = fmaf(bf16_lo(pa[2 * i]), ka.x, dot);
                dot = fmaf(bf16_hi(pa[2 * i]), ka.y, dot);
                dot = fmaf(bf16_lo(pa[2 * i + 1]), ka.z, dot);
                dot = fmaf(bf16_hi(pa[2 * i + 1]), ka.w, dot);
                dot = fmaf(bf16_lo(pb[2 * i]), kb.x, dot);
                dot = fmaf(bf16_hi(pb[2 * i]), kb.y, dot);
                dot = fmaf(bf16_lo(pb[2 * i + 1]), kb.z, dot);
                dot = fmaf(bf16_hi(pb[2 * i + 1]), kb.w, dot);
            }
        } else {
            // column sums of the warp's rows of each frame; lane l ends with column
            // 16c + l (l < 16) or D/2 + 16c + l - 16
            const int col = lane < 16 ? 16 * c + lane : HALF + 16 * c + (lane - 16);
            const bool in_lo = valid && f == f_lo;
#pragma unroll 1
            for (int side = straddle ? 1 : 0; side >= 0; --side) {
                const bool take = side == 0 ? in_lo : (valid && !in_lo);
                float v[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[2 * i] = take ? bf16_lo(pa[i]) : 0.0f;
                    v[2 * i + 1] = take ? bf16_hi(pa[i]) : 0.0f;
                    v[16 + 2 * i] = take ? bf16_lo(pb[i]) : 0.0f;
                    v[16 + 2 * i + 1] = take ? bf16_hi(pb[i]) : 0.0f;
                }
                kpart[D * side + col] = reduce_scatter32(v, lane);
            }
        }
    }
    if (sect == 2) return;
    const float nrm = sqrtf(ss);
    if (sect == 0) {
        const float qk = nrm * __ldcg(p.ks + static_cast<int64_t>(h) * p.F + f);
        const float gap = valid ? p.scale * (qk - dot) : 0.0f;
        if (valid) {
            p.bound[static_cast<int64_t>(h) * p.N + n] = p.scale * qk;
            if (p.qnorm) p.qnorm[static_cast<int64_t>(h) * p.N + n] = nrm;
        }
        const float g = warp_max(gap);
        if (lane == 0) atomicMax(p.gmax + h, __float_as_uint(fmaxf(g, 0.0f)));
    } else {
        const float m0 = warp_max(valid && f == f_lo ? nrm : 0.0f);
        const float m1 = warp_max(valid && f != f_lo ? nrm : 0.0f);
        if (lane == 0) {
            // non-negative floats order like their bit patterns
            atomicMax(p.kmax + static_cast<int64_t>(h) * p.F + f_lo, __float_as_uint(m0));
            if (straddle) atomicMax(p.kmax + static_cast<int64_t>(h) * p.F + f_lo + 1, __float_as_uint(m1));
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads, 1)
    fsa_prep_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const PrepParams p)
{
    using C = PrepCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw_u32);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::MISC_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 8);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_total = p.tiles_kv + p.m_tiles * (p.H * D / 256);
    const int KB = p.dm / C::BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_ACC_FULL), 1);
        mbar_init(bar(C::B_ACC_EMPTY), 8);  // one arrival per epilogue warp
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kPrepWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    WaitCtl wc;
    wc.abort = abort_flag;
    wc.err_word = p.stats ? &p.stats->error : nullptr;
    wc.err_site = p.stats ? &p.stats->timeout_site : nullptr;
    wc.limit = p.wait_limit;

    if (warp == kPrepWarpTma) {
        // ------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW);
            uint32_t g = 0;  // K steps issued by this CTA
            bool ok = true;
            for (int t = blockIdx.x; t < n_total && ok; t += gridDim.x) {
                int m, nt;
                prep_tile<D>(p, t, m, nt);
                for (int kb = 0; kb < KB; ++kb) {
                    const int s = static_cast<int>(g % C::NS);
                    if (!mbar_wait(bar(C::B_EMPTY + s), ((g / C::NS) & 1) ^ 1, wc, SITE_PREP_EMPTY)) {
                        ok = false;
                        break;
                    }
                    // rows of x past N are zero-filled (a ragged last row tile)
                    mbar_arrive_expect_tx(bar(C::B_FULL + s), C::STAGE_BYTES);
                    tma_load_2d(sbase + s * C::STAGE_BYTES, &tmX, kb * C::BK, m * C::BM, bar(C::B_FULL + s));
                    tma_load_2d(sbase + s * C::STAGE_BYTES + C::A_BYTES, &tmW, kb * C::BK, nt * C::BN,
                                bar(C::B_FULL + s));
                    ++g;
                }
            }
            // Every copy this thread issued must land before the CTA may exit.
            for (uint32_t u = (g > C::NS ? g - C::NS : 0); u < g; ++u)
                mbar_wait(bar(C::B_FULL + u % C::NS), (u / C::NS) & 1, wc, SITE_PREP_DRAIN, false);
        }
    } else if (warp == kPrepWarpMma) {
        // ------------------------------------------------------------- MMA issuer
        const bool leader = elect_one();
        const uint64_t d0 = smem_desc_sw128(sbase, 16, 1024);
        uint32_t g = 0;
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_total && ok; t += gridDim.x, ++it) {
            if (!mbar_wait(bar(C::B_ACC_EMPTY), (it & 1) ^ 1, wc, SITE_PREP_ACC_EMPTY)) break;
            tc_fence_after();
            for (int kb = 0; kb < KB; ++kb) {
                const int s = static_cast<int>(g % C::NS);
                if (!mbar_wait(bar(C::B_FULL + s), (g / C::NS) & 1, wc, SITE_PREP_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            // 16 bf16 = 32 B along the 128-byte swizzle row; rows 128 j.. of A
                            const uint64_t a = d0 + ((s * C::STAGE_BYTES + j * (C::A_BYTES / 2) + ks * 32) >> 4);
                            const uint64_t b = d0 + ((s * C::STAGE_BYTES + C::A_BYTES + ks * 32) >> 4);
                            mma_ss(tbase + 256u * j, a, b, C::IDESC, (kb > 0 || ks > 0) ? 1u : 0u);
                        }
                    tc_commit(bar(C::B_EMPTY + s));
                }
                __syncwarp();
                ++g;
            }
            if (!ok) break;
            if (leader) tc_commit(bar(C::B_ACC_FULL));
            __syncwarp();
        }
        // every MMA this thread issued completes before TMEM is released
        if (leader) tc_commit(bar(C::B_DRAIN));
        __syncwarp();
        mbar_wait(bar(C::B_DRAIN), 0, wc, SITE_PREP_DRAIN, false);
    } else {
        // ------------------------------------------------------------- epilogue
        // warp w reads TMEM lane quarter w % 4 of accumulator w / 4, its 256 / D heads in turn
        constexpr int HALF = D / 2;
        const int qd = warp & 3, j = warp >> 2;
        const uint32_t trow = tbase + (static_cast<uint32_t>(32 * qd) << 16) + 256u * j;
        float2* delta = reinterpret_cast<float2*>(sgen + C::DELTA_OFF);
        float2* rbase = reinterpret_cast<float2*>(sgen + C::RBASE_OFF) + 64 * warp;
        // delta[i][l] = rotary table row l, pair i (the table has at least 32 rows of D/2 pairs)
        for (int e = threadIdx.x; e < HALF * 32; e += 256) delta[(e % HALF) * 32 + e / HALF] = p.rope[e];
        asm volatile("bar.sync 1, 256;" ::: "memory");
        int it = 0;
        bool stats_done = false;
        for (int t = blockIdx.x; t < n_total; t += gridDim.x, ++it) {
            // Every epilogue warp calls prep_key_stats exactly once (here, or after the loop if it
            // left the loop early), so the named barriers inside it always match.
            if (t >= p.tiles_kv && !stats_done) {
                prep_key_stats<D>(p, threadIdx.x, wc);
                stats_done = true;
            }
            int m, nt;
            prep_tile<D>(p, t, m, nt);
            const int n_first = m * C::BM + 128 * j + 32 * qd;
            // loads that do not depend on the accumulators are issued before waiting for them
            const bool act = n_first < p.N;
            const int nn = act ? min(n_first + lane, p.N - 1) : 0;
            const float ri = p.rinv[nn];
            const float2 r0 = p.rope[static_cast<int64_t>(act ? n_first : 0) * HALF + lane];
            const float2 r1 = HALF > 32 ? p.rope[static_cast<int64_t>(act ? n_first : 0) * HALF + 32 + lane] : r0;
            if (!mbar_wait(bar(C::B_ACC_FULL), it & 1, wc, SITE_PREP_ACC_FULL)) break;
            tc_fence_after();
            __syncwarp();  // the previous tile's reads of rbase are done
            rbase[lane] = r0;
            if (HALF > 32) rbase[32 + lane] = r1;
            __syncwarp();
#pragma unroll 1
            for (int hh = 0; hh < C::BN / D && act; ++hh) {
                const int col0 = nt * C::BN + D * hh;  // first output column of the head
                const int sect = col0 / (p.H * D);
                const int h = col0 / D - sect * p.H;
                prep_epilogue<D>(p, trow + static_cast<uint32_t>(D * hh), sect, h, n_first, lane, ri, delta, rbase);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ACC_EMPTY));
        }
        // a CTA with no Q tile, or whose epilogue stopped early, still takes its share of the
        // key statistics and arrives at the grid barriers (after an abort without waiting)
        if (!stats_done) prep_key_stats<D>(p, threadIdx.x, wc);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPrepWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

// 1 / sqrt(mean(x^2) + eps) per token row, one warp per row, 16-byte loads.
__global__ void __launch_bounds__(256) rms_kernel(const uint16_t* __restrict__ x, int N, int dm, float eps,
                                                  float* __restrict__ rinv)
{
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const uint4* r = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row) * dm);
    float s = 0.0f;
    for (int i = lane; i < dm / 8; i += 32) {
        const uint4 u = __ldg(r + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = bf16_lo(w[k]), b = bf16_hi(w[k]);
            s = fmaf(a, a, s);
            s = fmaf(b, b, s);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) rinv[row] = 1.0f / sqrtf(s / static_cast<float>(dm) + eps);
}

}  // namespace

int prep_smem_bytes() { return PrepCfg::SMEM_BYTES; }

template <int D>
static int launch_prep_d(const PrepLaunch& L)
{
    static bool attr_done = false;  // per instantiation
    if (!attr_done) {
        if (cudaFuncSetAttribute(fsa_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PrepCfg::SMEM_BYTES) != cudaSuccess)
            return -3;
        attr_done = true;
    }
    const PrepParams& p = L.params;
    rms_kernel<<<(p.N + 7) / 8, 256, 0, L.stream>>>(L.x, p.N, p.dm, L.eps, p.rinv);
    if (cudaMemsetAsync(p.gsync, 0, 3 * sizeof(unsigned), L.stream) != cudaSuccess) return -3;
    // One CTA per SM, all resident at once (the grid barriers need it; a cooperative launch
    // refuses a grid that cannot be).
    const int total = p.tiles_kv + p.m_tiles * (p.H * D / 256);
    const int grid = total < L.sms ? total : L.sms;
    PrepParams pp = p;
    void* args[] = {const_cast<CUtensorMap*>(L.tmX), const_cast<CUtensorMap*>(L.tmW), &pp};
    if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fsa_prep_kernel<D>), dim3(grid), dim3(kPrepThreads),
                                    args, PrepCfg::SMEM_BYTES, L.stream) != cudaSuccess)
        return -3;
    return launch_status();
}

// Grid-barrier self test: every CTA meets at the prep kernel's grid barrier, whose target is
// the CTA count plus `missing`.  With missing = 0 the barrier opens; with missing = 1 it never
// does, and each CTA's waiting thread must give up after `limit` cycles, raise its CTA's abort
// flag and record FSA_ERR_TIMEOUT with the grid-barrier site.  result: [status, site, CTAs that
// saw their abort flag raised, arrivals counted].
__global__ void __launch_bounds__(256) fsa_selftest_grid_kernel(unsigned* counter, unsigned missing, long long limit,
                                                                int* result)
{
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    WaitCtl wc;
    wc.abort = &abort_flag;
    wc.err_word = result + 0;
    wc.err_site = result + 1;
    wc.limit = limit;
    grid_sync(counter, gridDim.x + missing, static_cast<int>(threadIdx.x), wc);
    __syncthreads();
    if (threadIdx.x == 0) {
        if (abort_flag) atomicAdd(result + 2, 1);
        if (blockIdx.x == 0) atomicMax(result + 3, static_cast<int>(ld_acquire_gpu(counter)));
    }
}

int launch_selftest_grid(long long limit, int ctas, int missing, unsigned* d_counter, int* d_result,
                         cudaStream_t stream)
{
    unsigned miss = static_cast<unsigned>(missing);
    void* args[] = {&d_counter, &miss, &limit, &d_result};
    // cooperative: every CTA is resident, as in the prep kernel, so an open barrier opens
    if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fsa_selftest_grid_kernel), dim3(ctas), dim3(256),
                                    args, 0, stream) != cudaSuccess)
        return -3;
    return launch_status();
}

int launch_prep(const PrepLaunch& L)
{
    if (L.D == 128) return launch_prep_d<128>(L);
    if (L.D == 64) return launch_prep_d<64>(L);
    return -2;
}

}  // namespace fsa
