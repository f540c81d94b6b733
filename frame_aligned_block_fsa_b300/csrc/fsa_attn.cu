// fsa_attn.cu -- frame-aligned block-sparse attention forward for B300 (sm_103a).
//
// Method: "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU" (aihot.vn).
//  * section "Xoa bo mat na", Fig. 3: blocks divide a frame's token range, so every key tile
//    of a query frame is fully inside the mask; the kernel walks the frame's key runs (the
//    window and, if outside it, the reference frame) in ONE softmax, with no mask predicate,
//    no padding of the key side and no second pass or merge;
//  * section "Giai phong Softmax", Fig. 4: on eligible heads the running max is replaced by
//    the per-row upper bound b_i = c ||q_i|| max ||k_j|| computed beforehand, so
//    p = exp(s - b_i) needs no rescale of the accumulator, and no tile depends on the one
//    before it; heads that fail the eligibility test take the running-max path inside the
//    same kernel.  Launches that run the running-max path alone use an instantiation without
//    the norm-bound loop (BOUND = false), so that loop does not shape its register allocation.
//
// B300 design: a persistent kernel, one CTA per SM, 12 warps.  The work list is every
// (head, frame, 128-row query tile); CTA b takes items b, b + G, b + 2G, ... (G CTAs), in
// head-major, frame-major order, so the CTAs that run at the same time share their heads'
// K and V in L2.  Every role walks the same item sequence and, per item, the frame's key runs
// in key tiles of at most NK (<= 128) keys (the last tile of a run may be narrower, a multiple
// of 16).  A tile counter g runs over all items of the CTA.
//
//   warps 0-7   softmax and epilogue, in two groups of four (warps 0-3, 4-7), one warp per TMEM
//               lane quarter: a thread owns one query row.  Every group takes every tile, its
//               16-key chunks c = group + 2j (j = 0..3), so the eight warps turn one tile into P
//               together, with equal shares.  On norm-bound items each thread keeps a part of its
//               row sum; on running-max items the groups also exchange their tile maxima through
//               shared memory.  (Two groups rather than three leave each SM sub-partition two
//               busy softmax warps beside its control warp, and up to 168 registers a thread.)
//               Norm-bound items read a tile's scores in two sets of 16 columns: the load of a
//               set's next chunk goes out as soon as the set is packed, so its TMEM latency
//               hides behind the other set's arithmetic.
//   warp 8      issues the S side (the warp runs the loop, one elected lane issues):
//                 Q(item)  -> TMEM by tcgen05.cp from shared memory (two Q slots, so the copy
//                             for the next item never touches the one in use)
//                 S(g)     = Q K(g)^T      A = Q from TMEM, B = K tile from shared memory
//   warp 9      issues the PV side:
//                 O       += P(g) V(g)     A = P from TMEM, B = V tile from shared memory
//               (the pipe takes an MMA only when it has room, so an issuing thread is held for
//               about as long as its MMAs run; with two issuers one does its bookkeeping while
//               the other feeds the pipe)
//   warps 10-11 TMA producers, one for Q and K, one for V: K(g) and V(g) go to slot g & 1 of a K
//               and a V ring (the slots of S buffer g & 1), each item's Q tile into its own
//               staging buffer.
//
// Tensor work: S has two TMEM buffers of 128 keys (tile g uses buffer g & 1), so while the
// softmax turns S(g) into P(g) the pipe computes S(g + 1) and PV(g - 1).  PV(g) is issued once
// P(g) is in TMEM; S(g + 2) goes into the same buffer once PV(g) is done (a commit of the PV
// issuer frees the buffer).  A 128-key tile carries 1024 cycles of tensor work, twice a 64-key
// one, against the same per-tile bookkeeping of the issuers (measured: 128-key tiles are the
// fastest in both modes).
//
// One O accumulator: the epilogue of item k (O / l -> out) runs in all eight softmax warps
// when the tile walk reaches item k + 1 (after they produced the P of its first tile), while
// the pipe computes S of item k + 1; the first PV of item k + 1 waits until the epilogue has
// read O out of TMEM.
//
// TMEM (512 columns): [Q slot 0: D/2][Q slot 1: D/2][S buffers 0-1: 128 each][O: D].
// P(g) overwrites S(g) in its buffer after the softmax has read it: the 8 bf16-pair columns of
// the 16 keys of chunk c go to the first 8 columns of that chunk, so each warp overwrites only
// columns it has read itself.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa_internal.h"
#include "fsa_ptx.cuh"

namespace fsa {

constexpr int kGroups = 2;                  // softmax warp groups
constexpr int kGroupWarps = 4;              // one warp per lane quarter
constexpr int kSoftWarps = kGroups * kGroupWarps;  // 8
constexpr int kAttnThreads = 32 * (kSoftWarps + 4);  // + two tcgen05 issuers and two TMA warps
constexpr int kWarpS = kSoftWarps, kWarpPV = kSoftWarps + 1, kWarpTmaK = kSoftWarps + 2, kWarpTmaV = kSoftWarps + 3;
constexpr int kNBuf = 2;                    // S buffers
constexpr int kBufShift = 1;                // log2(kNBuf): tile g uses buffer g & (kNBuf - 1), phase g >> kBufShift
constexpr int kBufCols = 128;               // TMEM columns (= keys) of an S buffer
// Group g takes the 16-key chunks c = g + 2j (j = 0..3) of every tile.  It hands P over in two
// steps: after its chunks j = 0, 1 (over both groups: the first kPassChunks chunks), then after
// j = 2, 3; the PV MMAs of the first step's keys start while the second step runs.
constexpr int kPassChunks = 4;
// Frames whose key runs are copied to shared memory when the kernel starts; larger plans
// read them from global memory.
constexpr int kSmemRunFrames = 256;

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int PANELS = D / 64;              // 64-element (128 B) swizzle panels of a row
    static constexpr int KV_PANEL = kBufCols * 128;    // 128 rows x 128 B
    static constexpr int SLOT_BYTES = PANELS * KV_PANEL;  // one K or V tile of up to 128 rows
    static constexpr int Q_PANEL = 128 * 128;          // 128 rows x 128 B
    static constexpr int Q_BYTES = PANELS * Q_PANEL;
    // K(g) and V(g) go to slot g & 1 of a K and a V ring, the slots of S buffer g & 1: the
    // commit that ends S(g) frees K slot g & 1, the one that ends PV(g) frees V slot g & 1.
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_BYTES;
    static constexpr int V_OFF = K_OFF + kNBuf * SLOT_BYTES;
    static constexpr int BAR_OFF = V_OFF + kNBuf * SLOT_BYTES;
    // barrier indices
    static constexpr int B_KFULL = 0;                  // kNBuf: K slot b landed
    static constexpr int B_VFULL = kNBuf;              // kNBuf: V slot b landed
    static constexpr int B_QFULL = 2 * kNBuf;          // the staged Q tile landed
    static constexpr int B_QEMPTY = B_QFULL + 1;       // its copy into TMEM is done
    static constexpr int B_SFULL = B_QEMPTY + 1;       // kNBuf: S in buffer b complete (K slot b free)
    // kNBuf: P of chunks 0-3 in buffer b written (the softmax's first step: chunks group and
    // group + 2 of both groups): kSoftWarps arrivals, one from every softmax warp
    static constexpr int B_PFULL = B_SFULL + kNBuf;
    // kNBuf: P of chunks 4-7 written (the second step), kSoftWarps arrivals
    static constexpr int B_PFULL2 = B_PFULL + kNBuf;
    static constexpr int B_OFULL = B_PFULL2 + kNBuf;   // the last PV of an item done: O final
    static constexpr int B_OFREE = B_OFULL + 1;        // the epilogue has read O (all softmax warps)
    static constexpr int B_BFREE = B_OFREE + 1;        // kNBuf: PV of buffer b's tile done (S buffer b and V
                                                       // slot b free)
    static constexpr int B_QDONE = B_BFREE + kNBuf;    // 2: the last S MMA of an item using Q slot s done
    static constexpr int B_DRAIN = B_QDONE + 2;        // 2: everything an issuer issued is done
    static constexpr int N_BARS = B_DRAIN + 2;
    // abort flag (+0), TMEM address (+4), per lane quarter: row-sum exchange counters (+8 .. +24),
    // tile-max exchange counters (+24 .. +40)
    static constexpr int MISC_OFF = BAR_OFF + 8 * N_BARS;
    static constexpr int MISC_BYTES = 48;
    // per item parity, group, row: a group's part of the row sum (epilogue)
    static constexpr int LSUM_OFF = (MISC_OFF + MISC_BYTES + 15) & ~15;
    static constexpr int LSUM_BYTES = 2 * kGroups * 128 * 4;
    // per exchange parity, group, row: a group's tile max (running-max tiles)
    static constexpr int MMAX_OFF = LSUM_OFF + LSUM_BYTES;
    static constexpr int MMAX_BYTES = 2 * kGroups * 128 * 4;
    static constexpr int RUNS_OFF = MMAX_OFF + MMAX_BYTES;
    // per softmax warp: 32 rows x 32 columns of out (fp32), rows 144 B apart so that both the
    // row-per-lane writes and the 8-lanes-per-row reads are free of bank conflicts
    static constexpr int OSTG_ROW = 32 * 4 + 16;
    static constexpr int OSTG_WARP = 32 * OSTG_ROW;
    static constexpr int OSTG_OFF = (RUNS_OFF + kSmemRunFrames * kRunStride * 4 + 15) & ~15;
    static constexpr int SMEM_USED = OSTG_OFF + kSoftWarps * OSTG_WARP;
    // room to align the buffers to 1024 B, and at least half of the SM's shared memory, so two
    // CTAs never share an SM (each takes all 512 TMEM columns)
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM: its 512 TMEM columns are not shared");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t t_q(int s) { return static_cast<uint32_t>(s * (D / 2)); }
    static constexpr uint32_t t_s(int b) { return static_cast<uint32_t>(D + kBufCols * b); }
    static constexpr uint32_t T_O = static_cast<uint32_t>(D + kBufCols * kNBuf);
    static_assert(D + kBufCols * kNBuf + D <= 512, "TMEM budget");
    static constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);
};

// wait sites (diagnostic codes in fsa_stats_t::timeout_site)
enum : int {
    SITE_PROD_EMPTY = 1, SITE_PROD_Q = 2, SITE_MMA_SLOT = 3, SITE_MMA_OFREE = 4, SITE_MMA_Q = 5, SITE_MMA_P = 6,
    SITE_SOFT_S = 7, SITE_SOFT_O = 8, SITE_DRAIN = 9, SITE_SELFTEST = 10, SITE_SOFT_X = 11
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kFltMin = 1.17549435e-38f;
constexpr float kUnderflowGap = 87.33654475055310898657f;  // 126 ln 2

// The key tiles of one CTA's items, in order.  An item is one 128-row query tile (h, f, qt);
// its keys are the runs of frame f (at most two: the window and the reference frame when it
// lies outside the window), cut into tiles of at most NK keys.  In the masked block variant an
// item is a 128-row tile of a query block on the padded sequence with one key run, read from
// its item table.  The kernel parameters are passed to every call instead of being held, so the
// iterator costs registers only for its position.
template <bool MASKED>
struct TileIter {
    int it;                          // current item index
    int local = -1;                  // items of this CTA begun so far, minus one
    int h = 0, row0 = 0, valid = 0;  // current item: head, first query token, valid rows
    int s0 = 0, l0 = 0, s1 = 0, lt = 0, pos = 0;  // runs (lt = total keys) and position

    __device__ TileIter() : it(static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x)) {}

    __device__ __forceinline__ bool load(const AttnParams& p, const int32_t* runs_tab)
    {
        it += static_cast<int>(gridDim.x);
        if (it >= p.total) {
            lt = pos = 0;
            return false;
        }
        ++local;
        h = it / p.per_head;
        const int loc = it - h * p.per_head;
        if constexpr (MASKED) {
            const int32_t* R = runs_tab + loc * kRunStride;
            row0 = R[kMaskItemRow];
            valid = min(128, p.N - row0);
            s0 = R[kMaskItemKey];
            l0 = R[kMaskItemLen];
            s1 = 0;
            lt = l0;
        } else {
            const int f = loc / p.n_qt;
            const int qt = loc - f * p.n_qt;
            row0 = f * p.T + qt * 128;
            valid = min(128, p.T - qt * 128);
            const int32_t* R = runs_tab + f * kRunStride;
            const int nr = R[0];
            s0 = R[1];
            l0 = R[2];
            s1 = nr > 1 ? R[3] : 0;
            lt = l0 + (nr > 1 ? R[4] : 0);
        }
        pos = 0;
        return true;
    }

    // The next tile: first key (token within the head), width, first / last tile of its item.
    __device__ __forceinline__ bool next(const AttnParams& p, const int32_t* runs_tab, int& start, int& width,
                                         bool& first, bool& last)
    {
        if (pos == lt && !load(p, runs_tab)) return false;
        first = pos == 0;
        if (pos < l0) {
            start = s0 + pos;
            width = min(p.NK, l0 - pos);
        } else {
            start = s1 + (pos - l0);
            width = min(p.NK, lt - pos);
        }
        pos += width;
        last = pos == lt;
        return true;
    }
};

// Bounded waits of the attention kernel.  The abort flag lives in shared memory and the limit and
// error words come from the kernel parameters, so a waiter keeps nothing in registers for them.
// A waiter that gives up raises the abort flag and records FSA_ERR_TIMEOUT and its site.
struct AttnWait {
    uint32_t abort_addr;

    __device__ __forceinline__ bool aborted() const
    {
        uint32_t v;
        asm volatile("ld.volatile.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(abort_addr) : "memory");
        return v != 0;
    }
    __device__ __noinline__ void fail(const AttnParams& p, int site) const
    {
        asm volatile("st.volatile.shared::cta.u32 [%0], %1;" ::"r"(abort_addr), "r"(1u) : "memory");
        if (p.stats) {
            atomicCAS(&p.stats->error, 0, -4 /* FSA_ERR_TIMEOUT */);
            atomicCAS(&p.stats->timeout_site, 0, site);
        }
    }
    // wait for the phase of the given parity of mbarrier `b`
    __device__ __forceinline__ bool bar(const AttnParams& p, uint32_t b, uint32_t parity, int site,
                                        bool honour_abort = true) const
    {
        if (mbar_test_wait(b, parity)) return true;
        const long long t0 = clock64();
        while (true) {
            if (mbar_try_wait(b, parity)) return true;
            if (honour_abort && aborted()) return false;
            if (clock64() - t0 > p.wait_limit) {
                fail(p, site);
                return false;
            }
        }
    }
    // wait until the shared counter at `addr` reaches `target`
    __device__ __forceinline__ bool counter(const AttnParams& p, uint32_t addr, uint32_t target, int site) const
    {
        if (static_cast<int>(ld_acquire_shared(addr) - target) >= 0) return true;
        const long long t0 = clock64();
        uint32_t nap = 16;
        while (true) {
            if (static_cast<int>(ld_acquire_shared(addr) - target) >= 0) return true;
            __nanosleep(nap);
            nap = min(nap * 2u, 256u);
            if (aborted()) return false;
            if (clock64() - t0 > p.wait_limit) {
                fail(p, site);
                return false;
            }
        }
    }
};

template <int D, bool MASKED, bool BOUND>
__global__ void __launch_bounds__(kAttnThreads, 1)
    fsa_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p)
{
    using C = AttnCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw_u32);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 4);
    uint32_t* counters = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // key runs of every frame (masked variant: the item table) into shared memory when they fit
    const bool runs_in_smem = p.n_tab <= kSmemRunFrames;
    int32_t* runs_s = reinterpret_cast<int32_t*>(sgen + C::RUNS_OFF);
    if (runs_in_smem)
        for (int i = threadIdx.x; i < p.n_tab * kRunStride; i += blockDim.x) runs_s[i] = p.runs[i];
    const int32_t* runs_tab = runs_in_smem ? runs_s : p.runs;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNBuf; ++b) {
            mbar_init(bar(C::B_KFULL + b), 1);
            mbar_init(bar(C::B_VFULL + b), 1);
        }
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QEMPTY), 1);
        for (int b = 0; b < kNBuf; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_PFULL + b), kSoftWarps);
            mbar_init(bar(C::B_PFULL2 + b), kSoftWarps);
        }
        mbar_init(bar(C::B_OFULL), 1);
        mbar_init(bar(C::B_OFREE), kSoftWarps);
        for (int b = 0; b < kNBuf; ++b) mbar_init(bar(C::B_BFREE + b), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_QDONE + i), 1);
            mbar_init(bar(C::B_DRAIN + i), 1);
        }
        for (int i = 0; i < 8; ++i) counters[i] = 0;
        *reinterpret_cast<volatile int*>(sgen + C::MISC_OFF) = 0;  // abort flag
        fence_mbar_init();
    }
    if (warp == kWarpS) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    const AttnWait wt{sbase + C::MISC_OFF};

    auto kslot = [&](int b) -> uint32_t { return sbase + C::K_OFF + b * C::SLOT_BYTES; };
    auto vslot = [&](int b) -> uint32_t { return sbase + C::V_OFF + b * C::SLOT_BYTES; };

    if (warp == kWarpTmaK || warp == kWarpTmaV) {
        // ------------------------------------------------------------- TMA producers
        // One warp loads Q and K, the other V, each waiting only on the barriers of its own
        // stream.  Rows past the tensor are zero-filled; rows past a narrower tile are loaded but
        // never read.
        if (lane == 0) {
            const bool is_k = warp == kWarpTmaK;
            tma_prefetch_desc(is_k ? &tmK : &tmV);
            if (is_k) tma_prefetch_desc(&tmQ);
            const uint64_t pol_kv = policy_evict_last();
            const uint64_t pol_q = policy_evict_first();
            const uint32_t kv_bytes = static_cast<uint32_t>(p.NK * D * 2);
            const CUtensorMap* map = is_k ? &tmK : &tmV;
            const uint32_t ring = is_k ? sbase + C::K_OFF : sbase + C::V_OFF;
            const int b_full = is_k ? C::B_KFULL : C::B_VFULL;
            // a slot is free once the tensor work that read it is done: S(g - 4) for K slot g & 3,
            // PV(g - 4) for V slot g & 3
            const int b_free = is_k ? C::B_SFULL : C::B_BFREE;
            TileIter<MASKED> it;
            int n = 0, nq = 0;  // tiles and Q tiles issued
            int start, width;
            bool first, last;
            while (it.next(p, runs_tab, start, width, first, last)) {
                const int hrow = it.h * p.N;
                if (is_k && first) {
                    // the item's Q tile, once the previous one has been copied into TMEM
                    if (!wt.bar(p, bar(C::B_QEMPTY), (nq & 1) ^ 1, SITE_PROD_Q)) break;
                    mbar_arrive_expect_tx(bar(C::B_QFULL), static_cast<uint32_t>(C::Q_BYTES));
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_2d_hint(sbase + C::Q_OFF + pn * C::Q_PANEL, &tmQ, pn * 64, hrow + it.row0,
                                         bar(C::B_QFULL), pol_q);
                    ++nq;
                }
                const int b = n & (kNBuf - 1);
                if (n >= kNBuf && !wt.bar(p, bar(b_free + b), ((n >> kBufShift) & 1) ^ 1, SITE_PROD_EMPTY)) break;
                mbar_arrive_expect_tx(bar(b_full + b), kv_bytes);
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_2d_hint(ring + b * C::SLOT_BYTES + pn * C::KV_PANEL, map, pn * 64, hrow + start,
                                     bar(b_full + b), pol_kv);
                ++n;
            }
            // Every copy this thread issued must land before the CTA may exit.
            if (nq > 0) wt.bar(p, bar(C::B_QFULL), (nq - 1) & 1, SITE_DRAIN, false);
            for (int u = n > kNBuf ? n - kNBuf : 0; u < n; ++u)
                wt.bar(p, bar(b_full + (u & (kNBuf - 1))), (u >> kBufShift) & 1, SITE_DRAIN, false);
        }
    } else if (warp == kWarpS) {
        // ------------------------------------------------------------- tcgen05 issuer: Q, S
        // The whole warp runs the loop, so the waits stay warp-uniform; one elected lane issues
        // every tcgen05 instruction (a commit tracks the work of its own thread).  The tests of
        // the next tile's barriers go out right after the first MMA of a tile, so their answers
        // are back while the pipe still has that tile's MMAs to run.
        const bool leader = elect_one();
        TileIter<MASKED> si;
        int nq = 0;  // Q tiles copied into TMEM
        bool ok = true;
        int start, width;
        bool first, last;
        bool more = si.next(p, runs_tab, start, width, first, last);
        bool k_seen = false, b_seen = true;  // readiness of tile x, tested ahead
        for (int x = 0; ok && more; ++x) {
            const int buf = x & (kNBuf - 1);
            const int qs = si.local & 1;
            const bool t_last = last;
            if (first) {
                // the Q slot was last read by item local - 2, whose last S must be done
                if (si.local >= 2 &&
                    !(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_QDONE + qs), ((si.local >> 1) & 1) ^ 1,
                                                          SITE_MMA_Q))))
                    break;
                if (!(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_QFULL), nq & 1, SITE_MMA_Q)))) break;
                tc_fence_after();
                const uint64_t d0 = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        tmem_cp_128x256b(tbase + C::t_q(qs) + ks * 8,
                                         d0 + static_cast<uint64_t>(((ks >> 2) * C::Q_PANEL + (ks & 3) * 32) >> 4));
                    tc_commit(bar(C::B_QEMPTY));
                }
                ++nq;
            }
            // S(x) overwrites the buffer of tile x - 4, whose PV must be done; K(x) must be in
            if (!__all_sync(0xffffffffu, b_seen) &&
                !(ok = __all_sync(0xffffffffu,
                                  wt.bar(p, bar(C::B_BFREE + buf), ((x >> kBufShift) & 1) ^ 1, SITE_MMA_P))))
                break;
            if (!__all_sync(0xffffffffu, k_seen) &&
                !(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_KFULL + buf), (x >> kBufShift) & 1, SITE_MMA_SLOT))))
                break;
            tc_fence_after();
            const uint64_t b0 = smem_desc_sw128(kslot(buf), 16, 1024);
            const uint32_t idesc = idesc_bf16_f32(128, width, false, false);
            const uint32_t tq = tbase + C::t_q(qs);
            if (leader) mma_ts(tbase + C::t_s(buf), tq, b0, idesc, 0u);
            {
                const int xn = x + 1, bn = xn & (kNBuf - 1);
                k_seen = mbar_test_wait(bar(C::B_KFULL + bn), (xn >> kBufShift) & 1);
                b_seen = xn < kNBuf || mbar_test_wait(bar(C::B_BFREE + bn), ((xn >> kBufShift) & 1) ^ 1);
            }
            if (leader) {
#pragma unroll
                for (int ks = 1; ks < D / 16; ++ks)
                    mma_ts(tbase + C::t_s(buf), tq + ks * 8,
                           b0 + static_cast<uint64_t>(((ks >> 2) * C::KV_PANEL + (ks & 3) * 32) >> 4), idesc, 1u);
                tc_commit(bar(C::B_SFULL + buf));
                if (t_last) tc_commit(bar(C::B_QDONE + qs));
            }
            __syncwarp();
            more = si.next(p, runs_tab, start, width, first, last);
        }
        // Every tcgen05 instruction this warp issued must complete before TMEM is released.
        if (leader) tc_commit(bar(C::B_DRAIN));
        __syncwarp();
        wt.bar(p, bar(C::B_DRAIN), 0, SITE_DRAIN, false);
        __syncwarp();
    } else if (warp == kWarpPV) {
        // ------------------------------------------------------------- tcgen05 issuer: PV
        const bool leader = elect_one();
        TileIter<MASKED> vi;
        int n_items = 0;
        long long n_pairs = 0;
        bool ok = true;
        int start, width;
        bool first, last;
        bool more = vi.next(p, runs_tab, start, width, first, last);
        bool p_seen = false, v_seen = false;  // readiness of tile g, tested ahead
        for (int g = 0; ok && more; ++g) {
            const int buf = g & (kNBuf - 1);
            const bool t_first = first, t_last = last;
            const int t_width = width;
            if (first) {
                // the epilogue of the previous item must have read O
                if (vi.local > 0 &&
                    !(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_OFREE), (vi.local - 1) & 1, SITE_MMA_OFREE))))
                    break;
            }
            if (!__all_sync(0xffffffffu, v_seen) &&
                !(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_VFULL + buf), (g >> kBufShift) & 1, SITE_MMA_SLOT))))
                break;
            if (!__all_sync(0xffffffffu, p_seen) &&
                !(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_PFULL + buf), (g >> kBufShift) & 1, SITE_MMA_P))))
                break;
            tc_fence_after();
            // O += P(g) V(g): A = P from the S buffer (16 keys = 8 columns per step)
            const uint64_t b0 = smem_desc_sw128(vslot(buf), C::KV_PANEL, 1024);
            if (leader)
                mma_ts(tbase + C::T_O, tbase + C::t_s(buf), b0, C::IDESC_O, t_first ? 0u : 1u);
            {
                const int gn = g + 1, bn = gn & (kNBuf - 1);
                p_seen = mbar_test_wait(bar(C::B_PFULL + bn), (gn >> kBufShift) & 1);
                v_seen = mbar_test_wait(bar(C::B_VFULL + bn), (gn >> kBufShift) & 1);
            }
            if (leader) {
#pragma unroll
                for (int ks = 1; ks < kPassChunks; ++ks)
                    if (ks < t_width / 16)
                        mma_ts(tbase + C::T_O, tbase + C::t_s(buf) + ks * 16,
                               b0 + static_cast<uint64_t>((ks * 16 * 128) >> 4), C::IDESC_O, 1u);
            }
            __syncwarp();
            // the last four chunks of P come from the softmax's second step (every tile's phase of
            // that barrier is waited for, so this thread never falls two phases behind)
            if (!(ok = __all_sync(0xffffffffu,
                                  wt.bar(p, bar(C::B_PFULL2 + buf), (g >> kBufShift) & 1, SITE_MMA_P))))
                break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int ks = kPassChunks; ks < kBufCols / 16; ++ks)
                    if (ks < t_width / 16)
                        mma_ts(tbase + C::T_O, tbase + C::t_s(buf) + ks * 16,
                               b0 + static_cast<uint64_t>((ks * 16 * 128) >> 4), C::IDESC_O, 1u);
                tc_commit(bar(C::B_BFREE + buf));
                if (t_last) tc_commit(bar(C::B_OFULL));
            }
            __syncwarp();
            // coverage: the (query row, key) pairs this item's tiles consumed
            n_pairs += static_cast<long long>(vi.valid) * t_width;
            n_items += t_last ? 1 : 0;
            more = vi.next(p, runs_tab, start, width, first, last);
        }
        if (p.stats && leader) {
            if (n_items > 0) atomicAdd(&p.stats->items_done, n_items);
            if (n_pairs > 0)
                atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats->pairs_visited),
                          static_cast<unsigned long long>(n_pairs));
        }
        if (leader) tc_commit(bar(C::B_DRAIN + 1));
        __syncwarp();
        wt.bar(p, bar(C::B_DRAIN + 1), 0, SITE_DRAIN, false);
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax + epilogue
        // Warp w: group w >> 2, lane quarter w & 3 (its 32 rows).  A thread owns one row of its
        // group's tiles, all of the tile's keys; in the epilogue each group takes a share of O's
        // columns.
        const int group = warp >> 2;
        const int quarter = warp & 3;
        const int row = 32 * quarter + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;

        // bound of this row and eligibility of the head of an item (prefetched one item ahead,
        // so the loads are in flight while the previous item runs)
        auto fetch = [&](int item, float& b, int& el) {
            b = 0.0f;
            el = 1;
            if (MASKED || item >= p.total) return;
            const int h = item / p.per_head;
            const int loc = item - h * p.per_head;
            const int f = loc / p.n_qt;
            const int qt = loc - f * p.n_qt;
            if (p.bound && row < min(128, p.T - qt * 128))
                b = __ldg(p.bound + static_cast<int64_t>(h) * p.N + f * p.T + qt * 128 + row);
            if (p.eligible) el = __ldg(p.eligible + h);
        };
        float nx_b;
        int nx_el;
        fetch(blockIdx.x, nx_b, nx_el);

        // current item: this row (h N + token), valid rows | bound flag << 8, bound, running state
        // m2: the reference of the exponentials on running-max items, mt: the row max (both in
        // log2 units of the logits)
        int grow = 0, flags = 0;
        float b_nat = 0.0f, m2 = -INFINITY, mt = -INFINITY, l = 0.0f;
        // the previous item, whose epilogue waits until the tile walk reaches the next item:
        // valid rows | bound flag << 8 | item << 9, or -1 for none
        int pv_grow = 0, pv_flags = -1;
        float pv_b = 0.0f, pv_m2 = 0.0f, pv_mt = 0.0f, pv_l = 0.0f;
        uint32_t n_mx = 0;   // tile-max exchanges done
        bool ok = true;

        // out = O / l for the rows of the previous item and this group's share of the columns
        // (16-column chunks [cb, ce)); lse (and the row max) by group 0.  The row sum is split
        // over the groups (each summed its own tiles); they exchange the parts first, and add
        // them in group order.  False on abort.
        auto epilogue = [&]() -> bool {
            const int item = pv_flags >> 9;
            const uint32_t ls_count = sbase + C::MISC_OFF + 8u + 4u * quarter;
            const uint32_t ls = sbase + C::LSUM_OFF + (item & 1) * (kGroups * 128 * 4) + 4u * row;
            st_shared_f32(ls + group * 512, pv_l);
            __syncwarp();
            if (lane == 0) red_release_shared_add(ls_count, 1u);
            if (!__all_sync(0xffffffffu,
                            wt.counter(p, ls_count, kGroups * static_cast<uint32_t>(item + 1), SITE_SOFT_X)))
                return false;
            float l_row = ld_shared_f32(ls);
#pragma unroll
            for (int j = 1; j < kGroups; ++j) l_row += ld_shared_f32(ls + 512 * j);
            // masked variant: a row without keys in this pass has l = 0: out 0, lse -inf
            const float inv_l = (MASKED && !(l_row > 0.0f)) ? 0.0f : 1.0f / l_row;
            const bool rvalid = row < (pv_flags & 0xff);
            const bool ub = (pv_flags >> 8) & 1;
            if (!__all_sync(0xffffffffu, wt.bar(p, bar(C::B_OFULL), item & 1, SITE_SOFT_O))) return false;
            tc_fence_after();
            const uint32_t tO = tbase + lane_off + C::T_O;
            // The group's D/2 columns in parts of 32: read from TMEM (this lane's row), scaled
            // into the warp's staging rows, then written with 8 lanes per row, so that each
            // store covers four whole 128-byte lines instead of touching 32 rows.  O is released
            // once its last part is in registers.
            constexpr int PARTS = D / 64;
            const int c0 = group * (D / 2);
            const int valid_rows = pv_flags & 0xff;
            float* out_w = p.out + static_cast<int64_t>(pv_grow - lane) * D + c0;  // the warp's row 0
            float* stg = reinterpret_cast<float*>(sgen + C::OSTG_OFF + warp * C::OSTG_WARP);
#pragma unroll
            for (int part = 0; part < PARTS; ++part) {
                float4* srow = reinterpret_cast<float4*>(stg + lane * (C::OSTG_ROW / 4));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float o[16];
                    tmem_ld_x16(tO + c0 + 32 * part + 16 * half, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) reg_fence(o[i]);
                    if (part == PARTS - 1 && half == 1) {
                        // every read of O by this warp is complete: the next item may overwrite O
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::B_OFREE));
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        srow[4 * half + e] = make_float4(o[4 * e] * inv_l, o[4 * e + 1] * inv_l,
                                                         o[4 * e + 2] * inv_l, o[4 * e + 3] * inv_l);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = 4 * k + (lane >> 3);
                    const float4 v = reinterpret_cast<const float4*>(stg + r * (C::OSTG_ROW / 4))[lane & 7];
                    // streaming stores: out is read by no one in this kernel, and lines that
                    // linger in L2 would displace the K and V tiles the CTAs re-read
                    if (32 * quarter + r < valid_rows)
                        __stcs(reinterpret_cast<float4*>(out_w + static_cast<int64_t>(r) * D + 32 * part) + (lane & 7), v);
                }
                __syncwarp();  // the staging rows are rewritten by the next part
            }
            if (group == 0) {
                const float m_nat = pv_mt * kLn2;
                bool under = false;
                if (rvalid) {
                    p.lse[pv_grow] = (ub ? pv_b : pv_m2 * kLn2) + logf(l_row);
                    if (p.rowmax) p.rowmax[pv_grow] = ub ? __int_as_float(0x7fc00000) : m_nat;
                    under = ub ? !(l_row >= kFltMin) : (p.bound != nullptr && pv_b - m_nat >= kUnderflowGap);
                }
                const unsigned ubits = __ballot_sync(0xffffffffu, under);
                if (p.stats && lane == 0 && ubits)
                    atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats->underflow_rows),
                              static_cast<unsigned long long>(__popc(ubits)));
            }
            return true;
        };

        // Walk the items; per item, every tile, this group's chunks of each.
        int g0 = 0;  // CTA tile index of the item's first tile
        for (int item = blockIdx.x, local = 0; ok && item < p.total; item += gridDim.x, ++local) {
            const int h = item / p.per_head;
            const int loc = item - h * p.per_head;
            // the item's key runs, cut into tiles of NK keys: n0 tiles of run 0 (the last of
            // them w0 keys), then n1 of run 1 (the last w1 keys)
            int n0, n1, w0, w1, valid, row0;
            // masked variant: this row's key interval [ja, jb) and the item's first key
            int ja = 0, jb = 0, kst = 0;
            if constexpr (MASKED) {
                const int32_t* R = runs_tab + loc * kRunStride;
                row0 = R[kMaskItemRow];
                kst = R[kMaskItemKey];
                n0 = R[kMaskItemLen] / p.NK;
                n1 = 0;
                w0 = p.NK;
                w1 = 0;
                valid = min(128, p.N - row0);
                if (row < valid) {
                    const int fi = (row0 + row) / p.T;
                    const int lo = max(0, fi - p.mask_w), hi = min(p.F - 1, fi + p.mask_w);
                    if (p.mask_pass == 0) {
                        ja = lo * p.T;
                        jb = (hi + 1) * p.T;
                    } else if (p.mask_ref < lo || p.mask_ref > hi) {
                        ja = p.mask_ref * p.T;
                        jb = ja + p.T;
                    }
                }
            } else {
                const int f = loc / p.n_qt;
                const int qt = loc - f * p.n_qt;
                const int32_t* R = runs_tab + f * kRunStride;
                const int l0 = R[2], l1 = R[0] > 1 ? R[4] : 0;
                n0 = (l0 + p.NK - 1) / p.NK;
                n1 = (l1 + p.NK - 1) / p.NK;
                w0 = l0 - (n0 - 1) * p.NK;
                w1 = l1 - (n1 - 1) * p.NK;
                valid = min(128, p.T - qt * 128);
                row0 = f * p.T + qt * 128;
            }
            const int n = n0 + n1;
            const bool use_bound = BOUND && !MASKED && p.mode == 0 && p.bound != nullptr && nx_el != 0;
            flags = valid | (use_bound ? 1 << 8 : 0);
            grow = h * p.N + row0 + row;
            b_nat = nx_b;
            fetch(item + static_cast<int>(gridDim.x), nx_b, nx_el);
            m2 = -INFINITY;
            mt = -INFINITY;
            l = 0.0f;
            if (p.stats && p.mode == 0 && !use_bound && warp == 0 && lane == 0 && loc == 0)
                atomicAdd(&p.stats->fallback_heads, 1);
            // Every group takes every tile: its 16-key chunks c = group + 2j (the split of the row
            // sum over the groups, and so its rounding, depends on the tile alone).  One loop per kind of item, so each stays small.
            if (use_bound) {
                const float nb2 = -b_nat * kLog2e;
                for (int t = 0; t < n; ++t) {
                    const int g = g0 + t;
                    const int width = t == n0 - 1 ? w0 : (t == n - 1 ? w1 : p.NK);
                    const int nch = width / 16;
                    const int buf = g & (kNBuf - 1);
                    const uint32_t tS = tbase + lane_off + C::t_s(buf);
                    const float c2 = row < (flags & 0xff) ? p.scale_log2 : 0.0f;
                    // the vote keeps the warp converged for the warp-collective TMEM accesses
                    if (!(ok = __all_sync(0xffffffffu,
                                          wt.bar(p, bar(C::B_SFULL + buf), (g >> kBufShift) & 1, SITE_SOFT_S))))
                        break;
                    tc_fence_after();
                    // p = 2^(s c2 - b log2 e) with the fixed bound, packed to bf16 over the first 8
                    // columns of each chunk just read; four partial sums of the fp32 weights.  Two
                    // steps of two chunks (group, group + 2; then group + 4, group + 6), each ending in
                    // a hand-over of its P.
                    const float2 c2x2 = make_float2(c2, c2), nb2x2 = make_float2(nb2, nb2);
                    float2 a01 = make_float2(0.0f, 0.0f), a23 = make_float2(0.0f, 0.0f);
                    const bool h0 = group < nch, h1 = group + 2 < nch, h2 = group + 4 < nch,
                               h3 = group + 6 < nch;
                    auto chunk = [&](float* sj, int c) {
                        uint32_t pk[8];
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float2 e = __ffma2_rn(make_float2(sj[i], sj[i + 1]), c2x2, nb2x2);
                            sj[i] = ex2(e.x);
                            sj[i + 1] = ex2(e.y);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(sj[2 * i], sj[2 * i + 1]);
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            a01 = __fadd2_rn(a01, make_float2(sj[i], sj[i + 1]));
                            a23 = __fadd2_rn(a23, make_float2(sj[i + 2], sj[i + 3]));
                        }
                        tmem_st_x8(tS + 16 * c, pk);
                    };
                    auto hand_over = [&](int b_full) {
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(b_full + buf));
                    };
                    // two 16-column register sets: the next chunk's load goes out as soon as
                    // its set is free, so its latency hides behind the other set's arithmetic
                    float r0[16], r1[16];
                    if (h0) tmem_ld_x16(tS + 16 * group, r0);
                    if (h1) tmem_ld_x16(tS + 16 * (group + 2), r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) { reg_fence(r0[i]); reg_fence(r1[i]); }
                    if (h0) chunk(r0, group);
                    if (h2) tmem_ld_x16(tS + 16 * (group + 4), r0);
                    if (h1) chunk(r1, group + 2);
                    if (h3) tmem_ld_x16(tS + 16 * (group + 6), r1);
                    hand_over(C::B_PFULL);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) { reg_fence(r0[i]); reg_fence(r1[i]); }
                    if (h2) chunk(r0, group + 4);
                    if (h3) chunk(r1, group + 6);
                    hand_over(C::B_PFULL2);
                    l += (a01.x + a01.y) + (a23.x + a23.y);
                    if (pv_flags >= 0) {
                        if (!(ok = epilogue())) break;
                        pv_flags = -1;
                    }
                }
            } else {
                for (int t = 0; t < n; ++t) {
                    const int g = g0 + t;
                    const int width = t == n0 - 1 ? w0 : (t == n - 1 ? w1 : p.NK);
                    const int nch = width / 16;
                    const int buf = g & (kNBuf - 1);
                    const uint32_t tS = tbase + lane_off + C::t_s(buf);
                    // masked variant: rows past the sequence have an empty key interval instead
                    const float c2 = (MASKED || row < (flags & 0xff)) ? p.scale_log2 : 0.0f;
                    // the vote keeps the warp converged for the warp-collective TMEM accesses
                    if (!(ok = __all_sync(0xffffffffu,
                                          wt.bar(p, bar(C::B_SFULL + buf), (g >> kBufShift) & 1, SITE_SOFT_S))))
                        break;
                    tc_fence_after();
                    // Running max, shared by all groups.  The groups exchange their tile maxima;
                    // the exponentials use a reference m2 that moves only when the row max passes
                    // it by more than 8 (so every p stays below 2^8), and only then is the row's
                    // accumulator rescaled.
                    const bool h0 = group < nch, h1 = group + 2 < nch, h2 = group + 4 < nch, h3 = group + 6 < nch;
                    float s[64];
                    if (h0) tmem_ld_x16(tS + 16 * group, s);
                    if (h1) tmem_ld_x16(tS + 16 * (group + 2), s + 16);
                    if (h2) tmem_ld_x16(tS + 16 * (group + 4), s + 32);
                    if (h3) tmem_ld_x16(tS + 16 * (group + 6), s + 48);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 64; ++i) reg_fence(s[i]);
                    if constexpr (MASKED) {
                        // mask predicates, on tiles that are not wholly inside the row's interval
                        const int j0 = kst + t * p.NK;
                        if (!(j0 >= ja && j0 + width <= jb)) {
                            const unsigned span = static_cast<unsigned>(jb - ja);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int cj = j0 + 16 * (group + 2 * j) - ja;
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    if (static_cast<unsigned>(cj + e) >= span) s[16 * j + e] = -INFINITY;
                            }
                        }
                    }
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j == 0 ? h0 : (j == 1 ? h1 : (j == 2 ? h2 : h3))) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) m4[e & 3] = fmaxf(m4[e & 3], s[16 * j + e]);
                        }
                    }
                    // exchange slots double-buffered by parity: a warp writes exchange n + 2's slot
                    // only after every partner has written n + 1's, i.e. after it read n's
                    const uint32_t mcount = sbase + C::MISC_OFF + 24u + 4u * quarter;
                    const uint32_t ms = sbase + C::MMAX_OFF + (n_mx & 1) * (kGroups * 128 * 4) + 4u * row;
                    st_shared_f32(ms + 512 * group, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
                    __syncwarp();
                    if (lane == 0) red_release_shared_add(mcount, 1u);
                    ++n_mx;
                    if (!(ok = __all_sync(0xffffffffu, wt.counter(p, mcount, kGroups * n_mx, SITE_SOFT_X)))) break;
                    float tmax = ld_shared_f32(ms);
#pragma unroll
                    for (int j = 1; j < kGroups; ++j) tmax = fmaxf(tmax, ld_shared_f32(ms + 512 * j));
                    const float m_tile = tmax * c2;
                    mt = fmaxf(mt, m_tile);
                    float alpha = 1.0f;
                    if (t == 0) {
                        m2 = m_tile;  // O and l start from zero: nothing to rescale
                    } else if (__any_sync(0xffffffffu, m_tile > m2 + 8.0f)) {
                        // O may be rescaled only once PV of the item's previous tile is done
                        if (!(ok = __all_sync(0xffffffffu, wt.bar(p, bar(C::B_BFREE + ((g - 1) & (kNBuf - 1))),
                                                                  ((g - 1) >> kBufShift) & 1, SITE_SOFT_O))))
                            break;
                        tc_fence_after();
                        const float m_new = m_tile > m2 + 8.0f ? m_tile : m2;
                        // (masked variant: a row with no key yet keeps m2 = -inf and alpha = 1)
                        alpha = (!MASKED || m_new > m2) ? ex2(m2 - m_new) : 1.0f;
                        m2 = m_new;
                        // this warp's share of the row's accumulator (the epilogue's column split)
                        constexpr int NCHO = D / 16;
                        const int cb = group * NCHO / kGroups, ce = (group + 1) * NCHO / kGroups;
                        const uint32_t tO = tbase + lane_off + C::T_O;
#pragma unroll 1
                        for (int c = cb; c < ce; ++c) {
                            float o[16];
                            tmem_ld_x16(tO + 16 * c, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                reg_fence(o[e]);
                                o[e] *= alpha;
                            }
                            tmem_st_x16(tO + 16 * c, o);
                        }
                    }
                    // masked variant: m2 = -inf only while every key of the row so far, this tile's
                    // included, is masked; their weights are 2^-inf = 0
                    const float nb2 = (MASKED && m2 == -INFINITY) ? 0.0f : -m2;
                    const float2 c2x2 = make_float2(c2, c2), nb2x2 = make_float2(nb2, nb2);
                    float2 a01 = make_float2(0.0f, 0.0f);  // two partial sums in one packed add
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j == 0 ? h0 : (j == 1 ? h1 : (j == 2 ? h2 : h3))) {
                            float* sj = s + 16 * j;
                            uint32_t pk[8];
#pragma unroll
                            for (int i = 0; i < 16; i += 2) {
                                const float2 e = __ffma2_rn(make_float2(sj[i], sj[i + 1]), c2x2, nb2x2);
                                sj[i] = ex2(e.x);
                                sj[i + 1] = ex2(e.y);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(sj[2 * i], sj[2 * i + 1]);
#pragma unroll
                            for (int i = 0; i < 16; i += 2) a01 = __fadd2_rn(a01, make_float2(sj[i], sj[i + 1]));
                            tmem_st_x8(tS + 16 * (group + 2 * j), pk);
                        }
                        if (j == 1) {
                            // chunks group and group + 2 are in TMEM: the first step is done
                            tmem_st_wait();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(C::B_PFULL + buf));
                        }
                    }
                    l = l * alpha + (a01.x + a01.y);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_PFULL2 + buf));
                    if (pv_flags >= 0) {
                        if (!(ok = epilogue())) break;
                        pv_flags = -1;
                    }
                }
            }
            if (!ok) break;
            pv_flags = flags | (local << 9);
            pv_b = b_nat;
            pv_m2 = m2;
            pv_mt = mt;
            pv_l = l;
            pv_grow = grow;
            g0 += n;
        }
        if (ok && pv_flags >= 0) ok = epilogue();
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpS) {
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

template <int D, bool MASKED, bool BOUND>
static int launch_attn(const AttnLaunch& L)
{
    using C = AttnCfg<D>;
    auto kern = fsa_attn_fwd_kernel<D, MASKED, BOUND>;
    static bool attr_done = false;  // per instantiation
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return -3;
        }
        attr_done = true;
    }
    if (L.params.total <= 0) return 0;
    const unsigned grid = static_cast<unsigned>(L.params.total < L.sms ? L.params.total : L.sms);
    kern<<<grid, kAttnThreads, C::SMEM_BYTES, L.stream>>>(*L.tmQ, *L.tmK, *L.tmV, L.params);
    return launch_status();
}

int attn_smem_bytes(int D)
{
    if (D == 64) return AttnCfg<64>::SMEM_BYTES;
    if (D == 128) return AttnCfg<128>::SMEM_BYTES;
    return -1;
}

int launch_attention(const AttnLaunch& L)
{
    static_assert(kMaxKeyTile == kBufCols, "one key tile fills an S buffer at most");
    if (L.params.NK < 16 || L.params.NK > kMaxKeyTile || L.params.NK % 16 != 0) return -2;
    if (L.masked && (L.params.mode != 1 || L.params.bound != nullptr || L.params.NK != kMaxKeyTile)) return -2;
    const bool bound = !L.masked && L.params.mode == 0;
    if (L.D == 64)
        return L.masked ? launch_attn<64, true, false>(L)
                        : (bound ? launch_attn<64, false, true>(L) : launch_attn<64, false, false>(L));
    if (L.D == 128)
        return L.masked ? launch_attn<128, true, false>(L)
                        : (bound ? launch_attn<128, false, true>(L) : launch_attn<128, false, false>(L));
    return -2;
}

// One warp per row of the [H][N] rows.  Rows whose window [f - w, f + w] (clipped) leaves out
// the reference frame: lse = log(e^lse + e^lse2) and out = e^(lse - lse') out + e^(lse2 - lse')
// out2; other rows keep the window pass's result.  A reference pass without keys for the row
// (lse2 = -inf) leaves it unchanged too.
__global__ void __launch_bounds__(256) masked_merge_kernel(float* __restrict__ out, float* __restrict__ lse,
                                                           const float* __restrict__ out2,
                                                           const float* __restrict__ lse2, int64_t rows, int N,
                                                           int T, int F, int w, int ref, int D)
{
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const int i = static_cast<int>(r % N);
    const int f = i / T;
    if (ref >= max(0, f - w) && ref <= min(F - 1, f + w)) return;
    const float l1 = lse[r], l2 = lse2[r];
    if (!(l2 > -INFINITY)) return;
    const float m = fmaxf(l1, l2);
    const float e1 = expf(l1 - m), e2 = expf(l2 - m);
    const float inv = 1.0f / (e1 + e2);
    const float a1 = e1 * inv, a2 = e2 * inv;
    float4* o = reinterpret_cast<float4*>(out + r * D);
    const float4* o2 = reinterpret_cast<const float4*>(out2 + r * D);
    for (int c = lane; c < D / 4; c += 32) {
        const float4 x = o[c], y = __ldg(o2 + c);
        o[c] = make_float4(a1 * x.x + a2 * y.x, a1 * x.y + a2 * y.y, a1 * x.z + a2 * y.z, a1 * x.w + a2 * y.w);
    }
    if (lane == 0) lse[r] = m + logf(e1 + e2);
}

int launch_masked_merge(float* out, float* lse, const float* out2, const float* lse2, int H, int N, int T, int F,
                        int w, int ref, int D, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(H) * N;
    if (rows == 0) return 0;
    const int64_t blocks = (rows + 7) / 8;
    masked_merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, lse, out2, lse2, rows, N, T, F, w,
                                                                          ref, D);
    return launch_status();
}

int launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream)
{
    fsa_selftest_wait_kernel<<<1, 32, 0, stream>>>(limit, d_status);
    return launch_status();
}

}  // namespace fsa
