// fsa_attn.cu -- frame-aligned block-sparse attention forward for B300 (sm_103a).
//
// Method: "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU" (aihot.vn).
//  * section "Xoa bo mat na", Fig. 3: blocks divide a frame's token range, so every key tile
//    of a query frame is fully inside the mask; the kernel walks the frame's key runs (the
//    window and, if outside it, the reference frame) in ONE softmax, with no mask predicate,
//    no padding of the key side and no second pass or merge;
//  * section "Giai phong Softmax", Fig. 4: on eligible heads the running max is replaced by
//    the per-row upper bound b_i = c ||q_i|| max ||k_j|| computed beforehand, so
//    p = exp(s - b_i) needs no rescale of the accumulator; heads that fail the eligibility
//    test take the running-max path inside the same kernel.
//
// B300 design (one CTA per SM, 10 warps):
//   warp 8      TMA producer: the CTA's two 128-row query tiles once, then K and V tiles of
//               NK keys through an NS-stage mbarrier ring (128-byte swizzled boxes).
//   warp 9      allocates TMEM and issues tcgen05.mma from one thread:
//                 S_j = Q_j K^T   (A, B from shared memory, fp32 accumulators in TMEM)
//                 O_j += P_j V    (A = P from TMEM, B = V from shared memory, MN-major)
//   warps 0-3   softmax + epilogue for query tile 0 (thread = row = TMEM lane)
//   warps 4-7   the same for query tile 1 (same frame, next 128 rows)
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D);
// P_j (bf16) overwrites the first NK/2 columns of S_j.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa_internal.h"
#include "fsa_ptx.cuh"

namespace fsa {

template <int D, int NK>
struct AttnCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(NK % 16 == 0 && NK >= 16 && NK <= kMaxKeyTile(D), "key tile");
    static constexpr int BM = 128;                      // query rows per tile (MMA M)
    static constexpr int PANELS = D / 64;               // 64-element (128 B) swizzle panels
    static constexpr int Q_PANEL_BYTES = BM * 128;
    static constexpr int Q_TILE_BYTES = BM * D * 2;
    static constexpr int KV_PANEL_BYTES = NK * 128;
    static constexpr int KV_TILE_BYTES = NK * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;  // K and V
    static constexpr int SMEM_LIMIT = 232448;              // max dynamic smem per block
    static constexpr int RESERVED = 256;                   // barriers + flags
    static constexpr int NS_FIT = (SMEM_LIMIT - 1024 - RESERVED - 2 * Q_TILE_BYTES) / STAGE_BYTES;
    static constexpr int NS = NS_FIT < 4 ? NS_FIT : 4;
    static_assert(NS >= 2, "pipeline depth");
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = 2 * Q_TILE_BYTES;
    static constexpr int V_OFF = K_OFF + NS * KV_TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + NS * KV_TILE_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + NS;
    static constexpr int B_KVEMPTY = B_VFULL + NS;
    static constexpr int B_SFULL = B_KVEMPTY + NS;  // 2
    static constexpr int B_PFULL = B_SFULL + 2;     // 2
    static constexpr int B_PVDONE = B_PFULL + 2;    // 2
    static constexpr int B_DRAIN = B_PVDONE + 2;
    static constexpr int N_BARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;  // abort flag, TMEM address
    static_assert(MISC_OFF + 16 <= BAR_OFF + RESERVED, "reserved area");
    static constexpr int SMEM_USED = 1024 + BAR_OFF + RESERVED;
    // At least half of the SM's shared memory, so two CTAs never share an SM and contend for
    // its 512 TMEM columns.
    static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(KV_PANEL_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    // TMEM columns per query tile j: S_j (fp32, NK columns) followed by P_j (bf16 pairs, NK/2
    // columns) inside a region of RS columns; then O_0 and O_1 (fp32, D columns each).
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t RS = ((NK + NK / 2) + 31) / 32 * 32;
    static_assert(2 * RS + 2 * D <= TMEM_COLS, "TMEM budget");
    static constexpr uint32_t t_s(int j) { return RS * j; }
    static constexpr uint32_t t_p(int j) { return RS * j + NK; }
    static constexpr uint32_t t_o(int j) { return 2 * RS + D * j; }
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, NK, false, false);
    static constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);
};

// wait sites (diagnostic codes in fsa_stats_t::timeout_site)
enum : int {
    SITE_PROD_EMPTY = 1, SITE_MMA_Q = 2, SITE_MMA_K = 3, SITE_MMA_PV = 4, SITE_MMA_V = 5,
    SITE_MMA_P = 6, SITE_SOFT_S = 7, SITE_SOFT_O = 8, SITE_DRAIN = 9, SITE_SELFTEST = 10
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kFltMin = 1.17549435e-38f;
constexpr float kUnderflowGap = 87.33654475055310898657f;  // 126 ln 2

// Loads `W` columns (W % 16 == 0) of this thread's TMEM lane into v (waits).
template <int W>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float* v)
{
#pragma unroll
    for (int c = 0; c < W / 16; ++c) tmem_ld_x16(taddr + 16 * c, v + 16 * c);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < W; ++i) reg_fence(v[i]);
}

template <int D, int NK>
__global__ void __launch_bounds__(320, 1)
    fsa_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p)
{
    using C = AttnCfg<D, NK>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw_u32);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::MISC_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.x / p.n_items;
    const int item = blockIdx.x - h * p.n_items;
    const int4 it = reinterpret_cast<const int4*>(p.items)[item];
    const int f = it.x, q_row0 = it.y, valid0 = it.z, valid1 = it.w;
    const int nq = valid1 > 0 ? 2 : 1;
    const int32_t* runs = p.runs + f * kRunStride;
    const int n_runs = runs[0];
    int n_tiles = 0;
    for (int r = 0; r < n_runs; ++r) n_tiles += runs[2 + 2 * r] / NK;
    const int64_t head_row0 = static_cast<int64_t>(h) * p.N;

    const bool use_bound = (p.mode == 0) && (p.bound != nullptr) &&
                           (p.eligible == nullptr || p.eligible[h] != 0);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar(C::B_SFULL + j), 1);
            mbar_init(bar(C::B_PFULL + j), 128);
            mbar_init(bar(C::B_PVDONE + j), 1);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.stats && item == 0 && p.mode == 0 && !use_bound) atomicAdd(&p.stats->fallback_heads, 1);
    }
    if (warp == 9) {
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

    if (warp == 8) {
        // ------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol_kv = policy_evict_last();
            mbar_arrive_expect_tx(bar(C::B_QFULL), static_cast<uint32_t>(nq * C::Q_TILE_BYTES));
            for (int j = 0; j < nq; ++j)
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_2d(sbase + C::Q_OFF + j * C::Q_TILE_BYTES + pn * C::Q_PANEL_BYTES, &tmQ,
                                pn * 64, static_cast<int>(head_row0 + q_row0 + j * 128), bar(C::B_QFULL));
            int t = 0;
            bool ok = true;
            for (int r = 0; r < n_runs && ok; ++r) {
                const int start = runs[1 + 2 * r];
                const int len = runs[2 + 2 * r];
                for (int k0 = 0; k0 < len; k0 += NK, ++t) {
                    const int st = t % C::NS;
                    if (!mbar_wait(bar(C::B_KVEMPTY + st), ((t / C::NS) & 1) ^ 1, wc, SITE_PROD_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const int row = static_cast<int>(head_row0 + start + k0);
                    mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::KV_TILE_BYTES);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_2d_hint(sbase + C::K_OFF + st * C::KV_TILE_BYTES + pn * C::KV_PANEL_BYTES,
                                         &tmK, pn * 64, row, bar(C::B_KFULL + st), pol_kv);
                    mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::KV_TILE_BYTES);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_2d_hint(sbase + C::V_OFF + st * C::KV_TILE_BYTES + pn * C::KV_PANEL_BYTES,
                                         &tmV, pn * 64, row, bar(C::B_VFULL + st), pol_kv);
                }
            }
            // Every copy this thread issued must land before the CTA may exit.
            mbar_wait(bar(C::B_QFULL), 0, wc, SITE_DRAIN, false);
            for (int u = (t > C::NS ? t - C::NS : 0); u < t; ++u) {
                mbar_wait(bar(C::B_KFULL + u % C::NS), (u / C::NS) & 1, wc, SITE_DRAIN, false);
                mbar_wait(bar(C::B_VFULL + u % C::NS), (u / C::NS) & 1, wc, SITE_DRAIN, false);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------- MMA issuer
        // Issue order per key tile t:  PV_0(t), S_0(t+1), PV_1(t), S_1(t+1).  While softmax 0
        // works on S_0(t+1) the tensor pipe runs PV_1(t) and S_1(t+1), and the other way round,
        // so the two query tiles keep the pipe busy in turn.  S_j(t+1) may overwrite S_j(t) as
        // soon as P_j(t) is signalled (its softmax has read S_j(t) by then); P_j lives in its
        // own columns, so it needs no wait for PV_j(t).
        if (lane == 0) {
            auto issue_s = [&](int j, uint32_t k_s) {
                const uint32_t q_s = sbase + C::Q_OFF + j * C::Q_TILE_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;  // 16 bf16 = 32 B inside the 128 B swizzle row
                    const uint64_t a = smem_desc_sw128(q_s + (ks >> 2) * C::Q_PANEL_BYTES + off, 16, 1024);
                    const uint64_t b = smem_desc_sw128(k_s + (ks >> 2) * C::KV_PANEL_BYTES + off, 16, 1024);
                    mma_ss(tbase + C::t_s(j), a, b, C::IDESC_S, ks > 0 ? 1u : 0u);
                }
                tc_commit(bar(C::B_SFULL + j));
            };
            bool ok = mbar_wait(bar(C::B_QFULL), 0, wc, SITE_MMA_Q);
            if (ok && n_tiles > 0) ok = mbar_wait(bar(C::B_KFULL), 0, wc, SITE_MMA_K);
            if (ok && n_tiles > 0) {
                tc_fence_after();
                for (int j = 0; j < nq; ++j) issue_s(j, sbase + C::K_OFF);
            }
            for (int t = 0; t < n_tiles && ok; ++t) {
                const int st = t % C::NS;
                const int st1 = (t + 1) % C::NS;
                const bool next = t + 1 < n_tiles;
                if (!(ok = mbar_wait(bar(C::B_VFULL + st), (t / C::NS) & 1, wc, SITE_MMA_V))) break;
                const uint32_t v_s = sbase + C::V_OFF + st * C::KV_TILE_BYTES;
                for (int j = 0; j < nq && ok; ++j) {
                    if (!(ok = mbar_wait(bar(C::B_PFULL + j), t & 1, wc, SITE_MMA_P))) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < NK / 16; ++ks) {
                        const uint64_t b = smem_desc_sw128(v_s + ks * 16 * 128, C::KV_PANEL_BYTES, 1024);
                        mma_ts(tbase + C::t_o(j), tbase + C::t_p(j) + ks * 8, b, C::IDESC_O,
                               (t > 0 || ks > 0) ? 1u : 0u);
                    }
                    tc_commit(bar(C::B_PVDONE + j));
                    if (next) {
                        if (j == 0) {
                            if (!(ok = mbar_wait(bar(C::B_KFULL + st1), ((t + 1) / C::NS) & 1, wc, SITE_MMA_K)))
                                break;
                            tc_fence_after();
                        }
                        issue_s(j, sbase + C::K_OFF + st1 * C::KV_TILE_BYTES);
                    }
                }
                if (!ok) break;
                tc_commit(bar(C::B_KVEMPTY + st));
            }
            // Every MMA this thread issued must complete before TMEM is released.
            tc_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0, wc, SITE_DRAIN, false);
        }
    } else {
        // ------------------------------------------------------------- softmax + epilogue
        const int j = warp >> 2;
        if (j < nq) {
            const int quarter = warp & 3;
            const int row = 32 * quarter + lane;
            const int valid = j == 0 ? valid0 : valid1;
            const bool rv = row < valid;
            const int64_t grow = head_row0 + q_row0 + 128 * j + row;
            const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
            const uint32_t tS = tbase + lane_off + C::t_s(j);
            const uint32_t tP = tbase + lane_off + C::t_p(j);
            const uint32_t tO = tbase + lane_off + C::t_o(j);
            const float c2 = rv ? p.scale_log2 : 0.0f;
            const float b_nat = (rv && p.bound) ? p.bound[grow] : 0.0f;
            const float nb2 = use_bound ? -b_nat * kLog2e : 0.0f;
            float m2 = -INFINITY;  // running max in log2 units (online path)
            float l = 0.0f;
            bool ok = true;
            for (int t = 0; t < n_tiles; ++t) {
                // the vote keeps the warp converged for the warp-collective TMEM accesses
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + j), t & 1, wc, SITE_SOFT_S)))) break;
                tc_fence_after();
                float s[NK];
                tmem_load_cols<NK>(tS, s);
                uint32_t pk[NK / 2];
                float lp[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // independent partial sums: short add chains
                float alpha = 1.0f, m_new = m2;
                if (use_bound) {
#pragma unroll
                    for (int e = 0; e < NK / 2; ++e) {
                        const float p0 = ex2(fmaf(s[2 * e], c2, nb2));
                        const float p1 = ex2(fmaf(s[2 * e + 1], c2, nb2));
                        pk[e] = pack_bf16x2(p0, p1);
                        lp[e & 3] += bf16_lo(pk[e]) + bf16_hi(pk[e]);  // normalise by the weights the MMA sees
                    }
                } else {
                    float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                    for (int i = 4; i < NK; ++i) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
                    m_new = fmaxf(m2, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2);
                    alpha = ex2(m2 - m_new);
#pragma unroll
                    for (int e = 0; e < NK / 2; ++e) {
                        const float p0 = ex2(fmaf(s[2 * e], c2, -m_new));
                        const float p1 = ex2(fmaf(s[2 * e + 1], c2, -m_new));
                        pk[e] = pack_bf16x2(p0, p1);
                        lp[e & 3] += bf16_lo(pk[e]) + bf16_hi(pk[e]);
                    }
                }
                l = l * alpha + ((lp[0] + lp[1]) + (lp[2] + lp[3]));
                if (t > 0) {
                    // P_j and O_j are free again once PV_j(t-1) has completed
                    if (!(ok = __all_sync(0xffffffffu,
                                          mbar_wait(bar(C::B_PVDONE + j), (t - 1) & 1, wc, SITE_SOFT_O))))
                        break;
                    tc_fence_after();
                    if (!use_bound && __any_sync(0xffffffffu, m_new > m2)) {
                        // running max moved: rescale the accumulator before PV_j(t) may start
#pragma unroll 1
                        for (int c = 0; c < D / 16; ++c) {
                            float o[16];
                            tmem_load_cols<16>(tO + 16 * c, o);
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] *= alpha;
                            tmem_st_x16(tO + 16 * c, o);
                        }
                    }
                }
                m2 = m_new;
#pragma unroll
                for (int c = 0; c < NK / 16; ++c) tmem_st_x8(tP + 8 * c, pk + 8 * c);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL + j));
            }
            if (ok && n_tiles > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PVDONE + j), (n_tiles - 1) & 1, wc, SITE_SOFT_O));
            if (ok) {
                tc_fence_after();
                const float inv_l = 1.0f / l;
                float* orow = p.out + grow * D;
#pragma unroll 1
                for (int c = 0; c < D / 16; ++c) {
                    float o[16];
                    tmem_load_cols<16>(tO + 16 * c, o);
                    if (rv) {
                        float4* dst = reinterpret_cast<float4*>(orow + 16 * c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(o[4 * e] * inv_l, o[4 * e + 1] * inv_l, o[4 * e + 2] * inv_l,
                                                 o[4 * e + 3] * inv_l);
                    }
                }
                const float m_nat = m2 * kLn2;
                bool under = false;
                if (rv) {
                    p.lse[grow] = (use_bound ? b_nat : m_nat) + logf(l);
                    if (p.rowmax) p.rowmax[grow] = use_bound ? __int_as_float(0x7fc00000) : m_nat;
                    under = use_bound ? !(l >= kFltMin) : (p.bound != nullptr && b_nat - m_nat >= kUnderflowGap);
                }
                const unsigned ub = __ballot_sync(0xffffffffu, under);
                if (p.stats && lane == 0 && ub)
                    atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats->underflow_rows),
                              static_cast<unsigned long long>(__popc(ub)));
            }
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

// Bounded-wait self test: one thread waits on a barrier that nothing arrives at.
__global__ void fsa_selftest_wait_kernel(long long limit, int* status)
{
    __shared__ __align__(8) uint64_t b;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&b), 1);
        fence_mbar_init();
        WaitCtl wc;
        wc.abort = &abort_flag;
        wc.err_word = status;
        wc.err_site = nullptr;
        wc.limit = limit;
        // phase 0 never completes: the wait must give up and report FSA_ERR_TIMEOUT
        const bool ok = mbar_wait(smem_u32(&b), 0, wc, SITE_SELFTEST);
        if (ok) atomicExch(status, 1);  // would mean the wait returned without an arrival
    }
}

template <int D, int NK>
static int launch_attn(const AttnLaunch& L)
{
    using C = AttnCfg<D, NK>;
    auto kern = fsa_attn_fwd_kernel<D, NK>;
    static bool attr_done = false;  // per instantiation
    if (!attr_done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
            cudaSuccess)
            return -3;
        attr_done = true;
    }
    const dim3 grid(static_cast<unsigned>(L.params.n_items) * static_cast<unsigned>(L.H));
    kern<<<grid, 320, C::SMEM_BYTES, L.stream>>>(*L.tmQ, *L.tmK, *L.tmV, L.params);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int attn_smem_bytes(int D, int NK)
{
#define FSA_SMEM_CASE(d, nk) \
    if (D == d && NK == nk) return AttnCfg<d, nk>::SMEM_BYTES;
    FSA_SMEM_CASE(64, 16) FSA_SMEM_CASE(64, 32) FSA_SMEM_CASE(64, 48) FSA_SMEM_CASE(64, 64)
    FSA_SMEM_CASE(64, 80) FSA_SMEM_CASE(64, 96) FSA_SMEM_CASE(64, 112) FSA_SMEM_CASE(64, 128)
    FSA_SMEM_CASE(128, 16) FSA_SMEM_CASE(128, 32) FSA_SMEM_CASE(128, 48) FSA_SMEM_CASE(128, 64) FSA_SMEM_CASE(128, 80)
#undef FSA_SMEM_CASE
    return -1;
}

int launch_attention(const AttnLaunch& L)
{
#define FSA_ATTN_CASE(d, nk) \
    if (L.D == d && L.NK == nk) return launch_attn<d, nk>(L);
    FSA_ATTN_CASE(64, 16) FSA_ATTN_CASE(64, 32) FSA_ATTN_CASE(64, 48) FSA_ATTN_CASE(64, 64)
    FSA_ATTN_CASE(64, 80) FSA_ATTN_CASE(64, 96) FSA_ATTN_CASE(64, 112) FSA_ATTN_CASE(64, 128)
    FSA_ATTN_CASE(128, 16) FSA_ATTN_CASE(128, 32) FSA_ATTN_CASE(128, 48) FSA_ATTN_CASE(128, 64) FSA_ATTN_CASE(128, 80)
#undef FSA_ATTN_CASE
    return -2;
}

int launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream)
{
    fsa_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit, d_status);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace fsa
