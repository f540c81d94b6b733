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
// B300 design (one CTA per SM, 18 warps, two 128-row query tiles j = 0, 1 of one frame):
//   warps 0-7   query tile 0: per key tile the softmax, at the end the epilogue.  A thread
//               owns one row (= TMEM lane); the two warps of a lane quarter (w and w + 4)
//               split the key tile's 16-column chunks (even / odd), so a row's
//               exponentials run in two warps at once.
//   warps 8-15  the same for query tile 1
//   warp 16     TMA producer: the two query tiles once, then K and V tiles of up to NK keys
//               through an NS-stage mbarrier ring (128-byte swizzled boxes)
//   warp 17     allocates TMEM and issues tcgen05.mma (the warp runs the loop, one elected
//               lane issues):
//                 S_j  = Q_j K^T   (A = Q_j, B = K tile, both from shared memory)
//                 O_j += P_j V     (A = P_j from TMEM, B = V tile from shared memory, MN-major)
//
// Each query tile has two S buffers in TMEM, so the MMAs run two key tiles ahead of the
// softmax: S_j(t+2) is issued right after PV_j(t), into the buffer PV_j(t) has just read P_j(t)
// from.  The softmax therefore finds S_j(t+1) ready when it finishes tile t, and the chain
// "softmax, hand-off, MMAs, hand-off back" no longer sets the pace; the tensor pipe and the
// exponentials do.  (The tensor pipe takes MMAs from a very short queue, so an issuing thread
// is blocked for about as long as its MMAs take; with one S buffer per tile the pipe idled
// for every hand-off.)  Q stays in shared memory to leave TMEM for the second buffer.
//
// TMEM (512 columns): per query tile j a 256-column region
//   [S_j buffer 0: NK fp32][S_j buffer 1: NK fp32][O_j: D fp32].
// P_j(t) overwrites S_j(t) in its buffer after the softmax has read it: the 8 bf16-pair
// columns of the 16 keys of S chunk c go to the first 8 columns of that chunk, so each warp
// overwrites only columns it has read itself.  S_j(t+2) is issued after PV_j(t) by the same
// thread, and the tensor pipe executes one thread's MMAs in issue order, so PV_j(t) has read
// P_j(t) before S_j(t+2) overwrites it.
//
// Key tiles: each key run (a whole number of frames) is cut into tiles of NK keys and one
// last narrower tile of the remaining len mod NK keys (a multiple of 16, since T is).  Every
// tile is fully inside the mask; a narrower tile is an MMA of smaller N (S) or K (PV).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa_internal.h"
#include "fsa_ptx.cuh"

namespace fsa {

constexpr int kAttnThreads = 576;  // 16 softmax warps, the TMA warp, the MMA warp
constexpr int kWarpTma = 16, kWarpMma = 17;

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
    static constexpr int LSUM_BYTES = 2 * 2 * 128 * 4;     // row-sum halves (epilogue)
    static constexpr int NS_FIT =
        (SMEM_LIMIT - 1024 - RESERVED - LSUM_BYTES - 2 * 2 * 2 * 128 * 4 - 2 * Q_TILE_BYTES) / STAGE_BYTES;
    static constexpr int NS = NS_FIT < 6 ? NS_FIT : 6;
    static_assert(NS >= 3, "pipeline depth: two key tiles ahead of the one being read");
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = 2 * Q_TILE_BYTES;
    static constexpr int V_OFF = K_OFF + NS * KV_TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + NS * KV_TILE_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_KVFULL = 1;                // NS: K and V of a stage landed
    static constexpr int B_KVEMPTY = B_KVFULL + NS;   // NS: the MMAs reading a stage are done
    static constexpr int B_SFULL = B_KVEMPTY + NS;    // 4: S_j in buffer b complete (index 2 j + b)
    static constexpr int B_PVDONE = B_SFULL + 4;      // 2: PV_j complete
    // 4: P_j of a key tile in buffer b in TMEM (index 2 j + b, 8 arrivals).  One barrier per
    // buffer: the softmax can finish key tile t+1 before the MMA warp has waited for tile t,
    // but never tile t+2, so each barrier is at most one phase ahead of its waiter.
    static constexpr int B_PFULL = B_PVDONE + 2;
    static constexpr int B_DRAIN = B_PFULL + 4;
    static constexpr int N_BARS = B_DRAIN + 1;
    // abort flag (+0), TMEM address (+8), row-sum exchange counters (+16, +20), row-max
    // exchange counters per (query tile, lane quarter) (+24 .. +56)
    static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
    static_assert(MISC_OFF + 56 <= BAR_OFF + RESERVED, "reserved area");
    // per query tile, per column half, per row: the half's partial row sum (epilogue)
    static constexpr int LSUM_OFF = BAR_OFF + RESERVED;
    // per key-tile parity, query tile, column half, row: the half's tile max (running-max path)
    static constexpr int MMAX_OFF = LSUM_OFF + LSUM_BYTES;
    static constexpr int MMAX_BYTES = 2 * 2 * 2 * 128 * 4;
    static constexpr int SMEM_USED = 1024 + MMAX_OFF + MMAX_BYTES;
    // At least half of the SM's shared memory, so two CTAs never share an SM and contend for
    // its 512 TMEM columns.
    static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(KV_PANEL_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t REGION = 256;
    static_assert(2 * NK + D <= static_cast<int>(REGION), "TMEM budget");
    static constexpr uint32_t t_s(int j, int b) { return REGION * j + NK * b; }  // chunk c's P at + 16 c
    static constexpr uint32_t t_o(int j) { return REGION * j + 2 * NK; }
    static constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);
};

// wait sites (diagnostic codes in fsa_stats_t::timeout_site)
enum : int {
    SITE_PROD_EMPTY = 1, SITE_MMA_Q = 2, SITE_MMA_K = 3, SITE_MMA_P = 6, SITE_SOFT_S = 7, SITE_SOFT_O = 8,
    SITE_DRAIN = 9, SITE_SELFTEST = 10
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

// Walks a query frame's key runs in tiles of at most NK keys: (first key, width).  The runs
// (at most kMaxRuns) are read once into registers, so that stepping costs no memory access.
template <int NK>
struct KeyTiles {
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0, l0 = 0, l1 = 0, l2 = 0, l3 = 0;
    int r = 0, k0 = 0;
    __device__ explicit KeyTiles(const int32_t* rr)
    {
        static_assert(kMaxRuns == 4, "one register pair per run");
        const int n = rr[0];
        s0 = rr[1];
        l0 = rr[2];
        if (n > 1) { s1 = rr[3]; l1 = rr[4]; }
        if (n > 2) { s2 = rr[5]; l2 = rr[6]; }
        if (n > 3) { s3 = rr[7]; l3 = rr[8]; }
    }
    __device__ __forceinline__ void next(int& start, int& width)
    {
        const int len = r == 0 ? l0 : (r == 1 ? l1 : (r == 2 ? l2 : l3));
        const int base = r == 0 ? s0 : (r == 1 ? s1 : (r == 2 ? s2 : s3));
        start = base + k0;
        width = min(NK, len - k0);
        k0 += width;
        if (k0 == len) {
            k0 = 0;
            ++r;
        }
    }
};

template <int D, int NK>
__global__ void __launch_bounds__(kAttnThreads, 1)
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
    uint32_t* xcount = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 16);
    // xcount[j] counts the row-sum halves of query tile j written to shared memory
    auto xcount_addr = [&](int j) -> uint32_t { return sbase + C::MISC_OFF + 16u + 4u * static_cast<uint32_t>(j); };

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
    for (int r = 0; r < n_runs; ++r) n_tiles += (runs[2 + 2 * r] + NK - 1) / NK;
    const int64_t head_row0 = static_cast<int64_t>(h) * p.N;

    const bool use_bound = (p.mode == 0) && (p.bound != nullptr) &&
                           (p.eligible == nullptr || p.eligible[h] != 0);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(C::B_SFULL + i), 1);
        for (int i = 0; i < 8; ++i) xcount[2 + i] = 0;
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar(C::B_PVDONE + j), 1);
            mbar_init(bar(C::B_PFULL + 2 * j), 8);  // one arrival per softmax warp of the tile
            mbar_init(bar(C::B_PFULL + 2 * j + 1), 8);
            xcount[j] = 0;
        }
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.stats && item == 0 && p.mode == 0 && !use_bound) atomicAdd(&p.stats->fallback_heads, 1);
    }
    if (warp == kWarpMma) {
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

    if (warp == kWarpTma) {
        // ------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol_kv = policy_evict_last();
            // Both query tiles in full (rows past the tensor are zero-filled; rows past the
            // frame are computed but never stored).
            mbar_arrive_expect_tx(bar(C::B_QFULL), static_cast<uint32_t>(nq * C::Q_TILE_BYTES));
            for (int j = 0; j < nq; ++j)
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_2d(sbase + C::Q_OFF + j * C::Q_TILE_BYTES + pn * C::Q_PANEL_BYTES, &tmQ, pn * 64,
                                static_cast<int>(head_row0 + q_row0 + j * 128), bar(C::B_QFULL));
            KeyTiles<NK> tiles(runs);
            int t = 0;
            for (; t < n_tiles; ++t) {
                const int st = t % C::NS;
                if (!mbar_wait(bar(C::B_KVEMPTY + st), ((t / C::NS) & 1) ^ 1, wc, SITE_PROD_EMPTY)) break;
                int start, width;
                tiles.next(start, width);
                // A narrower last tile still loads a full box: the rows past it are never read
                // by the MMAs (rows past the tensor are zero-filled).
                const int row = static_cast<int>(head_row0 + start);
                mbar_arrive_expect_tx(bar(C::B_KVFULL + st), 2 * C::KV_TILE_BYTES);
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_2d_hint(sbase + C::K_OFF + st * C::KV_TILE_BYTES + pn * C::KV_PANEL_BYTES, &tmK,
                                     pn * 64, row, bar(C::B_KVFULL + st), pol_kv);
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_2d_hint(sbase + C::V_OFF + st * C::KV_TILE_BYTES + pn * C::KV_PANEL_BYTES, &tmV,
                                     pn * 64, row, bar(C::B_KVFULL + st), pol_kv);
            }
            // Every copy this thread issued must land before the CTA may exit.
            mbar_wait(bar(C::B_QFULL), 0, wc, SITE_DRAIN, false);
            for (int u = (t > C::NS ? t - C::NS : 0); u < t; ++u)
                mbar_wait(bar(C::B_KVFULL + u % C::NS), (u / C::NS) & 1, wc, SITE_DRAIN, false);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------- MMA issuer
        // Prologue: S_j(0) into buffer 0 and S_j(1) into buffer 1 of every query tile j.  Per
        // key tile t, for j = 0, 1: once softmax j has put P_j(t) into buffer t % 2, PV_j(t),
        // then S_j(t+2) into the same buffer (the pipe runs one thread's MMAs in order).
        // PVDONE_j is committed after every PV on running-max heads (the softmax rescales O_j
        // only once PV_j(t-1) is done) and after the last PV on norm-bound heads.
        //
        // The whole warp runs this loop, so the waits and the descriptor arithmetic stay
        // warp-uniform; one elected lane issues every tcgen05.mma and tcgen05.commit (a commit
        // tracks the MMAs of its own thread, so the same lane issues all of them).
        const bool leader = elect_one();
        // Descriptor bases; moving the start address by b bytes adds b >> 4 to the descriptor.
        const uint64_t dq = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);
        const uint64_t dk = smem_desc_sw128(sbase + C::K_OFF, 16, 1024);
        const uint64_t dv = smem_desc_sw128(sbase + C::V_OFF, C::KV_PANEL_BYTES, 1024);
        // S_j = Q_j K^T into buffer buf; `probe` runs after the first MMA is queued, so that the
        // answer of an mbarrier test it issues is back by the time the group is queued.
        auto issue_s = [&](int j, int buf, int st, int width, auto&& probe) {
            const uint64_t a0 = dq + static_cast<uint64_t>((j * C::Q_TILE_BYTES) >> 4);
            const uint64_t b0 = dk + static_cast<uint64_t>((st * C::KV_TILE_BYTES) >> 4);
            const uint32_t idesc = idesc_bf16_f32(128, width, false, false);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                if (ks == 1) probe();
                // 16 bf16 = 32 B inside the 128 B swizzle row; a new 64-column panel every 4 steps
                const uint32_t qo = ((ks >> 2) * C::Q_PANEL_BYTES + (ks & 3) * 32) >> 4;
                const uint32_t ko = ((ks >> 2) * C::KV_PANEL_BYTES + (ks & 3) * 32) >> 4;
                if (leader) mma_ss(tbase + C::t_s(j, buf), a0 + qo, b0 + ko, idesc, ks > 0 ? 1u : 0u);
            }
            if (leader) tc_commit(bar(C::B_SFULL + 2 * j + buf));
            __syncwarp();
        };
        auto no_probe = [] {};
        auto issue_pv = [&](int j, int buf, int st, int width, bool first, bool commit) {
            const uint64_t b0 = dv + static_cast<uint64_t>((st * C::KV_TILE_BYTES) >> 4);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < NK / 16; ++ks)
                    if (ks < width / 16)
                        mma_ts(tbase + C::t_o(j), tbase + C::t_s(j, buf) + ks * 16, b0 + ((ks * 16 * 128) >> 4),
                               C::IDESC_O, (!first || ks > 0) ? 1u : 0u);
                if (commit) tc_commit(bar(C::B_PVDONE + j));
            }
            __syncwarp();
        };
        // An mbarrier test answers only after a long round trip while shared memory is busy,
        // so readiness is tested early (the answer `seen`) and waited for only when it was no.
        auto stage_test = [&](int t) { return mbar_test_wait(bar(C::B_KVFULL + t % C::NS), (t / C::NS) & 1); };
        auto stage_wait = [&](int t, bool seen) -> bool {
            if (__all_sync(0xffffffffu, seen)) return true;
            return __all_sync(0xffffffffu, mbar_wait(bar(C::B_KVFULL + t % C::NS), (t / C::NS) & 1, wc, SITE_MMA_K));
        };
        auto p_test = [&](int j, int t) { return mbar_test_wait(bar(C::B_PFULL + 2 * j + (t & 1)), (t >> 1) & 1); };
        auto p_wait = [&](int j, int t, bool seen) -> bool {
            if (__all_sync(0xffffffffu, seen)) return true;
            return __all_sync(0xffffffffu, mbar_wait(bar(C::B_PFULL + 2 * j + (t & 1)), (t >> 1) & 1, wc, SITE_MMA_P));
        };
        // widths of tiles t, t+1, t+2 (w_cur, w_1, w_2)
        KeyTiles<NK> tiles(runs);
        int start, w_cur = 0, w_1 = 0, w_2 = 0;
        bool ok = n_tiles > 0;
        if (ok) {
            tiles.next(start, w_cur);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_QFULL), 0, wc, SITE_MMA_Q));
        }
        if (ok) ok = stage_wait(0, false);
        if (ok) {
            tc_fence_after();
            for (int j = 0; j < nq; ++j) issue_s(j, 0, 0, w_cur, no_probe);
        }
        if (ok && n_tiles > 1) {
            tiles.next(start, w_1);
            if ((ok = stage_wait(1, false))) {
                tc_fence_after();
                for (int j = 0; j < nq; ++j) issue_s(j, 1, 1, w_1, no_probe);
            }
        }
        bool p_seen0 = false, p_seen1 = false;  // early answers: P_0(t), P_1(t) ready
        bool st_seen = n_tiles > 2 && ok && stage_test(2);  // early answer: tile t+2's stage landed
        // Loop state of key tile t: width of tile t+2 (w_2), read in the previous iteration so
        // that the next group's bookkeeping runs while MMAs of the current group are queued.
        bool ahead = n_tiles > 2;
        if (ahead) tiles.next(start, w_2);
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int st = t % C::NS;
            const int buf = t & 1;
            const bool last = t + 1 == n_tiles;
            const bool pv_commit = last || !use_bound;
            bool st_next = false;
            bool ahead_next = false;
            int w_3 = 0;
            // the work of the next key tile's loop head, done between MMAs of the last group
            auto advance = [&] {
                p_seen0 = t + 1 < n_tiles && p_test(0, t + 1);
                st_next = t + 3 < n_tiles && stage_test(t + 3);
                ahead_next = t + 3 < n_tiles;
                if (ahead_next) tiles.next(start, w_3);
            };
            // query tile 0
            if (!(ok = p_wait(0, t, p_seen0))) break;
            tc_fence_after();
            issue_pv(0, buf, st, w_cur, t == 0, pv_commit);
            if (ahead) {
                if (!(ok = stage_wait(t + 2, st_seen))) break;
                tc_fence_after();
            }
            auto probe0 = [&] {
                if (nq > 1)
                    p_seen1 = p_test(1, t);
                else
                    advance();
            };
            if (ahead)
                issue_s(0, buf, (t + 2) % C::NS, w_2, probe0);
            else
                probe0();
            // query tile 1
            if (nq > 1) {
                if (!(ok = p_wait(1, t, p_seen1))) break;
                tc_fence_after();
                issue_pv(1, buf, st, w_cur, t == 0, pv_commit);
                if (ahead)
                    issue_s(1, buf, (t + 2) % C::NS, w_2, advance);
                else
                    advance();
            }
            st_seen = st_next;
            ahead = ahead_next;
            w_cur = w_1;
            w_1 = w_2;
            w_2 = w_3;
            if (leader) tc_commit(bar(C::B_KVEMPTY + st));
            __syncwarp();
        }
        // Every MMA this warp issued must complete before TMEM is released.
        if (leader) tc_commit(bar(C::B_DRAIN));
        __syncwarp();
        mbar_wait(bar(C::B_DRAIN), 0, wc, SITE_DRAIN, false);
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax + epilogue
        const int j = warp >> 3;
        if (j < nq) {
            const int quarter = warp & 3;
            const int hf = (warp >> 2) & 1;  // this warp's chunks: c = 2 i + hf
            const int row = 32 * quarter + lane;
            const int valid = j == 0 ? valid0 : valid1;
            const bool rv = row < valid;
            const int64_t grow = head_row0 + q_row0 + 128 * j + row;
            const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
            const uint32_t tO = tbase + lane_off + C::t_o(j) + hf * (D / 2);  // this warp's half of O
            constexpr int OWN = (NK / 16 + 1) / 2;  // most chunks a warp owns
            const float c2 = rv ? p.scale_log2 : 0.0f;
            const float b_nat = (rv && p.bound) ? p.bound[grow] : 0.0f;
            const float nb2 = use_bound ? -b_nat * kLog2e : 0.0f;
            float m2 = -INFINITY;  // running max in log2 units (online path)
            float l = 0.0f;        // sum of this warp's weights of the row
            bool ok = true;
            KeyTiles<NK> tiles(runs);
            for (int t = 0; t < n_tiles; ++t) {
                int start, width;
                tiles.next(start, width);
                const int nch = width / 16;  // 16-column chunks of this tile
                const int buf = t & 1;
                const uint32_t tS = tbase + lane_off + C::t_s(j, buf);
                // the vote keeps the warp converged for the warp-collective TMEM accesses
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + 2 * j + buf), (t >> 1) & 1, wc,
                                                             SITE_SOFT_S))))
                    break;
                tc_fence_after();
                float s[16 * OWN];  // own chunks, compact
                uint32_t pk[8 * OWN];
#pragma unroll
                for (int i = 0; i < OWN; ++i)
                    if (2 * i + hf < nch) tmem_ld_x16(tS + 16 * (2 * i + hf), s + 16 * i);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16 * OWN; ++i) reg_fence(s[i]);
                // Two packed partial sums of the fp32 weights (short add chains).
                float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                float alpha = 1.0f, m_new = m2;
                float2 off = make_float2(nb2, nb2);
                if (!use_bound) {
                    // The running max over the whole row.  The two warps of the row exchange
                    // the maxima of their own chunks through shared memory: reading the other
                    // warp's chunks from TMEM could race with its P being written over them.
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < OWN; ++i) {
                        if (2 * i + hf < nch) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) mx[e & 3] = fmaxf(mx[e & 3], s[16 * i + e]);
                        }
                    }
                    const float mine = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                    // slots double-buffered by key-tile parity: a warp writes tile t+2's slot only
                    // after its partner has written tile t+1's, i.e. after it read tile t's
                    float* mslot = reinterpret_cast<float*>(sgen + C::MMAX_OFF) + (((t & 1) * 2 + j) * 2) * 128;
                    mslot[hf * 128 + row] = mine;
                    __syncwarp();
                    const uint32_t xa = sbase + C::MISC_OFF + 24u + 4u * static_cast<uint32_t>(4 * j + quarter);
                    if (lane == 0) red_release_shared_add(xa, 1u);
                    if (!(ok = __all_sync(0xffffffffu,
                                          counter_wait(xa, 2u * static_cast<uint32_t>(t + 1), wc, SITE_SOFT_S))))
                        break;
                    const float theirs = mslot[(1 - hf) * 128 + row];
                    m_new = fmaxf(m2, fmaxf(mine, theirs) * c2);
                    alpha = ex2(m2 - m_new);
                    off = make_float2(-m_new, -m_new);
                }
                const float2 cc = make_float2(c2, c2);
#pragma unroll
                for (int i = 0; i < OWN; ++i) {
                    if (2 * i + hf < nch) {
#pragma unroll
                        for (int e = 8 * i; e < 8 * i + 8; ++e) {
                            const float2 x = ffma2(make_float2(s[2 * e], s[2 * e + 1]), cc, off);
                            const float p0 = ex2(x.x);
                            const float p1 = ex2(x.y);
                            pk[e] = pack_bf16x2(p0, p1);
                            acc[e & 1] = fadd2(acc[e & 1], make_float2(p0, p1));
                        }
                    }
                }
                l = l * alpha + ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y));
                if (!use_bound && t > 0) {
                    // O_j may be rescaled only once PV_j(t-1) is done (committed every tile here)
                    if (!(ok = __all_sync(0xffffffffu,
                                          mbar_wait(bar(C::B_PVDONE + j), (t - 1) & 1, wc, SITE_SOFT_O))))
                        break;
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, m_new > m2)) {
                        // running max moved: rescale this warp's half of the accumulator before
                        // PV_j(t) may start
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
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
                for (int i = 0; i < OWN; ++i)
                    if (2 * i + hf < nch) tmem_st_x8(tS + 16 * (2 * i + hf), pk + 8 * i);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + 2 * j + buf));
            }
            // the last PV: phase n_tiles - 1 on running-max heads (every PV committed), the
            // only phase 0 on norm-bound heads
            if (ok && n_tiles > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PVDONE + j), use_bound ? 0 : (n_tiles - 1) & 1, wc,
                                                       SITE_SOFT_O));
            // The row sum is split over the two warps of the row: exchange the halves.
            float* lsum = reinterpret_cast<float*>(sgen + C::LSUM_OFF) + (2 * j) * 128;
            lsum[hf * 128 + row] = l;
            __syncwarp();
            if (lane == 0) red_release_shared_add(xcount_addr(j), 1u);
            if (ok) ok = __all_sync(0xffffffffu, counter_wait(xcount_addr(j), 8u, wc, SITE_SOFT_O));
            if (ok) {
                tc_fence_after();
                const float l_row = l + lsum[(1 - hf) * 128 + row];
                const float inv_l = 1.0f / l_row;
                float* orow = p.out + grow * D + hf * (D / 2);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
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
                if (hf == 0) {
                    const float m_nat = m2 * kLn2;
                    bool under = false;
                    if (rv) {
                        p.lse[grow] = (use_bound ? b_nat : m_nat) + logf(l_row);
                        if (p.rowmax) p.rowmax[grow] = use_bound ? __int_as_float(0x7fc00000) : m_nat;
                        under = use_bound ? !(l_row >= kFltMin)
                                          : (p.bound != nullptr && b_nat - m_nat >= kUnderflowGap);
                    }
                    const unsigned ub = __ballot_sync(0xffffffffu, under);
                    if (p.stats && lane == 0 && ub)
                        atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats->underflow_rows),
                                  static_cast<unsigned long long>(__popc(ub)));
                }
            }
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
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
    kern<<<grid, kAttnThreads, C::SMEM_BYTES, L.stream>>>(*L.tmQ, *L.tmK, *L.tmV, L.params);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

#define FSA_FOR_EACH_TILE(X) \
    X(64, 16) X(64, 32) X(64, 48) X(64, 64) X(128, 16) X(128, 32) X(128, 48) X(128, 64)

int attn_smem_bytes(int D, int NK)
{
#define FSA_SMEM_CASE(d, nk) \
    if (D == d && NK == nk) return AttnCfg<d, nk>::SMEM_BYTES;
    FSA_FOR_EACH_TILE(FSA_SMEM_CASE)
#undef FSA_SMEM_CASE
    return -1;
}

int launch_attention(const AttnLaunch& L)
{
#define FSA_ATTN_CASE(d, nk) \
    if (L.D == d && L.NK == nk) return launch_attn<d, nk>(L);
    FSA_FOR_EACH_TILE(FSA_ATTN_CASE)
#undef FSA_ATTN_CASE
    return -2;
}

int launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream)
{
    fsa_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit, d_status);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace fsa
