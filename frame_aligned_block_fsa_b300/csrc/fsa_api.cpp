// fsa_api.cpp -- the C ABI: argument checks, the frame-aligned block plan, device data,
// tensor maps and kernel launches.  See include/fsa.h for the contract of every call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "fsa.h"
#include "fsa_internal.h"

using fsa::kMaxRuns;
using fsa::kRunStride;

struct fsa_plan_s {
    int F = 0, T = 0, w = 0, ref = 0, block = 0;
    int64_t N = 0;
    std::vector<int32_t> row_ptr, col_idx;  // block CSR
    std::vector<int32_t> runs;              // [F][kRunStride], tokens within a head
    float tau = 64.0f;
    int key_tile = 0;                       // 0 = automatic
    int center_keys = 0;                    // 1: mean-centred key norms in the bound
    std::mutex mu;
    // device data, created on first device use
    int device = -1;
    int32_t* d_runs = nullptr;
    // norms workspace, grown on demand (capacities in elements)
    int64_t cap_qnorm = 0, cap_bound = 0, cap_kmax = 0, cap_ksum = 0, cap_gmax = 0, cap_elig = 0;
    int64_t cap_psum = 0, cap_pmax = 0, cap_tickets = 0, cap_mu = 0, cap_htickets = 0;
    float* d_psum = nullptr;
    float* d_pmax = nullptr;
    unsigned* d_tickets = nullptr;
    bool tickets_fresh = false;  // newly allocated: zero them on the next norms launch
    float* d_mu = nullptr;       // [H][D] head key means (centred keys)
    unsigned* d_htickets = nullptr;
    // fsa_prep workspace
    int64_t cap_rinv = 0, cap_kpart = 0, cap_ks = 0, cap_kbar = 0, cap_gsync = 0;
    int rope_d = 0;               // head dim the rotary table was built for
    unsigned* d_gsync = nullptr;  // grid-barrier counters of the prep kernel
    float* d_rinv = nullptr;
    float* d_kpart = nullptr;
    float* d_ks = nullptr;
    float* d_kbar = nullptr;
    float2* d_rope = nullptr;    // [N][64] (cos, sin), built once per plan
    int sms = 0;
    float* d_qnorm = nullptr;
    float* d_bound = nullptr;
    float* d_kmax = nullptr;
    float* d_ksum = nullptr;
    unsigned* d_gmax = nullptr;
    uint8_t* d_elig = nullptr;
    // fsa_forward_host: device copies of the problem, three streams and per-chunk events
    int64_t cap_in = 0, cap_out = 0, cap_lse = 0;  // elements
    uint16_t* d_hq = nullptr;
    uint16_t* d_hk = nullptr;
    uint16_t* d_hv = nullptr;
    float* d_hout = nullptr;
    float* d_hlse = nullptr;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> ev;                     // [2 * chunks + 1]
    // fsa_forward_masked: item tables of the last block size used (window pass, reference
    // pass) and the reference pass's results
    int mask_block = 0;
    int mask_n_win = 0, mask_n_ref = 0;              // items per head
    int32_t* d_mask_win = nullptr;
    int32_t* d_mask_ref = nullptr;
    int64_t cap_out2 = 0, cap_lse2 = 0;
    float* d_out2 = nullptr;
    float* d_lse2 = nullptr;
};

namespace {

thread_local int g_last_cuda_error = 0;

}  // namespace

void fsa::note_cuda_error(int code) { g_last_cuda_error = code; }

int fsa::launch_status()
{
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return 0;
    note_cuda_error(e);
    return -3;
}

namespace {

constexpr int kDriverErrorBase = 100000;  // driver (CUresult) codes are reported offset by this
constexpr long long kDefaultWaitLimit = 4000000000LL;  // SM clock cycles (about 2 s)

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return FSA_OK;
    fsa::note_cuda_error(e);
    return FSA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


int check_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FSA_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return FSA_ERR_CUDA;
    if (major != 10 || minor != 3) return FSA_ERR_UNSUPPORTED;  // built for sm_103a only
    return FSA_OK;
}

template <typename T>
int upload(T** dst, const std::vector<T>& src)
{
    if (cudaMalloc(reinterpret_cast<void**>(dst), std::max<size_t>(1, src.size()) * sizeof(T)) != cudaSuccess)
        return FSA_ERR_CUDA;
    if (!src.empty() && cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
        return FSA_ERR_CUDA;
    return FSA_OK;
}

// First device use: check the device, upload the key runs and read the SM count.
int ensure_device(fsa_plan_s* P)
{
    int rc = check_device();
    if (rc != FSA_OK) return rc;
    int dev = -1;
    cudaGetDevice(&dev);
    if (P->device == dev) return FSA_OK;
    if (P->device != -1) return FSA_ERR_INVALID_ARG;  // a plan serves one device
    if ((rc = upload(&P->d_runs, P->runs)) != FSA_OK) return rc;
    if (cudaDeviceGetAttribute(&P->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FSA_ERR_CUDA;
    P->device = dev;
    return FSA_OK;
}

template <typename T>
int grow(T** p, int64_t* cap, int64_t need)
{
    if (*cap >= need) return FSA_OK;
    if (*p) cudaFree(*p);
    *p = nullptr;
    *cap = 0;
    if (cudaMalloc(reinterpret_cast<void**>(p), static_cast<size_t>(need) * sizeof(T)) != cudaSuccess)
        return FSA_ERR_CUDA;
    *cap = need;
    return FSA_OK;
}

int ensure_workspace(fsa_plan_s* P, int H, int D)
{
    const int64_t hn = static_cast<int64_t>(H) * P->N;
    const int64_t hf = static_cast<int64_t>(H) * P->F;
    int rc;
    if ((rc = grow(&P->d_qnorm, &P->cap_qnorm, hn)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_bound, &P->cap_bound, hn)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_kmax, &P->cap_kmax, hf)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_ksum, &P->cap_ksum, hf * D)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_gmax, &P->cap_gmax, static_cast<int64_t>(H))) != FSA_OK) return rc;
    const int64_t chunks = fsa::norms_key_chunks(P->T);
    if ((rc = grow(&P->d_psum, &P->cap_psum, hf * chunks * D)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_pmax, &P->cap_pmax, hf * chunks)) != FSA_OK) return rc;
    const int64_t had = P->cap_tickets, had_h = P->cap_htickets;
    if ((rc = grow(&P->d_tickets, &P->cap_tickets, hf)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_htickets, &P->cap_htickets, 2 * static_cast<int64_t>(H))) != FSA_OK) return rc;
    if (P->cap_tickets != had || P->cap_htickets != had_h) P->tickets_fresh = true;
    if ((rc = grow(&P->d_mu, &P->cap_mu, static_cast<int64_t>(H) * D)) != FSA_OK) return rc;
    return grow(&P->d_elig, &P->cap_elig, static_cast<int64_t>(H));
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 [rows][D] row-major, boxes of 64 columns (128 bytes, the swizzle span) x box_rows.
int make_tensor_map(CUtensorMap* m, const void* base, int64_t rows, int D, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc) return FSA_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) return FSA_OK;
    fsa::note_cuda_error(kDriverErrorBase + static_cast<int>(r));
    return FSA_ERR_CUDA;
}

int check_shape(const fsa_plan_s* P, int H, int D)
{
    if (!P || H < 0) return FSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(H) * P->N >= (int64_t(1) << 31)) return FSA_ERR_INVALID_ARG;
    return FSA_OK;
}

int run_norms(fsa_plan_s* P, const uint16_t* q, const uint16_t* k, int H, int D, float* qnorm, float* kmax,
              float* bound, uint8_t* eligible, cudaStream_t stream)
{
    fsa::NormsLaunch L;
    L.q = q;
    L.k = k;
    L.H = H;
    L.D = D;
    L.F = P->F;
    L.T = P->T;
    L.N = static_cast<int>(P->N);
    L.runs = P->d_runs;
    L.scale = 1.0f / std::sqrt(static_cast<float>(D));
    L.tau = P->tau;
    L.qnorm = qnorm;
    L.kmax = kmax ? kmax : P->d_kmax;
    L.ksum = P->d_ksum;
    L.part_sum = P->d_psum;
    L.part_max = P->d_pmax;
    L.tickets = P->d_tickets;
    if (P->tickets_fresh) {
        if (cudaMemsetAsync(P->d_tickets, 0, static_cast<size_t>(P->cap_tickets) * sizeof(unsigned), stream) !=
                cudaSuccess ||
            cudaMemsetAsync(P->d_htickets, 0, static_cast<size_t>(P->cap_htickets) * sizeof(unsigned), stream) !=
                cudaSuccess)
            return FSA_ERR_CUDA;
        P->tickets_fresh = false;
    }
    L.center = P->center_keys;
    L.mu = P->d_mu;
    L.htickets = P->d_htickets;
    L.bound = bound ? bound : P->d_bound;
    L.gmax = P->d_gmax;
    L.eligible = eligible ? eligible : P->d_elig;
    L.stream = stream;
    const int rc = fsa::launch_norms(L);
    return rc == 0 ? FSA_OK : (rc == -2 ? FSA_ERR_UNSUPPORTED : FSA_ERR_CUDA);
}

// The attention step on device tensors; the caller holds the plan lock and has checked the
// arguments.  Runs the norms into the plan workspace first when norm_bound has no bound.
int forward_locked(fsa_plan_s* P, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse,
                   int H, int D, int NK, int mode, const float* bound, const uint8_t* eligible, float* rowmax,
                   fsa_stats_t* dev_stats, cudaStream_t st)
{
    int rc;
    if (mode == FSA_MODE_NORM_BOUND && bound == nullptr) {
        if ((rc = ensure_workspace(P, H, D)) != FSA_OK) return rc;
        if ((rc = run_norms(P, q, k, H, D, nullptr, nullptr, nullptr, nullptr, st)) != FSA_OK) return rc;
        bound = P->d_bound;
        eligible = P->d_elig;
    }
    const int64_t rows = static_cast<int64_t>(H) * P->N;
    CUtensorMap mq, mk, mv;
    if ((rc = make_tensor_map(&mq, q, rows, D, 128)) != FSA_OK) return rc;
    if ((rc = make_tensor_map(&mk, k, rows, D, NK)) != FSA_OK) return rc;
    if ((rc = make_tensor_map(&mv, v, rows, D, NK)) != FSA_OK) return rc;
    fsa::AttnLaunch L;
    L.D = D;
    L.H = H;
    L.masked = false;
    L.sms = P->sms;
    L.tmQ = &mq;
    L.tmK = &mk;
    L.tmV = &mv;
    L.stream = st;
    fsa::AttnParams& a = L.params;
    a.runs = P->d_runs;
    a.n_tab = P->F;
    a.F = P->F;
    a.T = P->T;
    a.N = static_cast<int>(P->N);
    a.n_qt = (P->T + 127) / 128;
    a.per_head = P->F * a.n_qt;
    a.total = H * a.per_head;
    a.NK = NK;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    a.mode = mode;
    a.bound = bound;
    a.eligible = eligible;
    a.out = out;
    a.lse = lse;
    a.rowmax = rowmax;
    a.stats = dev_stats;
    a.wait_limit = kDefaultWaitLimit;
    a.mask_w = a.mask_ref = a.mask_pass = 0;
    rc = fsa::launch_attention(L);
    return rc == 0 ? FSA_OK : (rc == -2 ? FSA_ERR_UNSUPPORTED : FSA_ERR_CUDA);
}

// Work items of the masked block variant with blocks of B tokens, one table per pass, the same
// for every head.  Query and key blocks of B tokens tile the sequence padded to a multiple of B.
// A query block takes every key block that meets the union of its rows' key intervals: the
// windows of its frames (one interval, pass 0) and, when the window of at least one of its
// frames leaves it out, the reference frame (pass 1).  Each 128-row tile of a query block that
// holds a real row is one item: [first row, first key, keys, 0, 0].
void masked_items(const fsa_plan_s* P, int B, std::vector<int32_t>& win, std::vector<int32_t>& refp)
{
    const int64_t N = P->N, T = P->T, F = P->F, w = P->w, r = P->ref;
    win.clear();
    refp.clear();
    const int64_t r0 = (r * T / B) * B, r1 = ((r + 1) * T + B - 1) / B * B;
    for (int64_t q0 = 0; q0 < N; q0 += B) {
        const int64_t q1 = std::min<int64_t>(N, q0 + B);
        const int64_t fa = q0 / T, fb = (q1 - 1) / T;
        const int64_t lo = std::max<int64_t>(0, fa - w), hi = std::min<int64_t>(F - 1, fb + w);
        const int64_t k0 = (lo * T / B) * B, k1 = ((hi + 1) * T + B - 1) / B * B;
        const bool need_ref = !(fb - w <= r && r <= fa + w);
        for (int64_t t0 = q0; t0 < q1; t0 += 128) {
            const int32_t a[kRunStride] = {static_cast<int32_t>(t0), static_cast<int32_t>(k0),
                                           static_cast<int32_t>(k1 - k0), 0, 0};
            win.insert(win.end(), a, a + kRunStride);
            if (need_ref) {
                const int32_t b[kRunStride] = {static_cast<int32_t>(t0), static_cast<int32_t>(r0),
                                               static_cast<int32_t>(r1 - r0), 0, 0};
                refp.insert(refp.end(), b, b + kRunStride);
            }
        }
    }
}

constexpr float kPrepEps = 1e-6f;           // RMS-norm epsilon
constexpr double kPrepRopeBase = 10000.0;   // rotary base

// Workspace of fsa_prep: 1/rms per token, K column partials, per-query-frame key statistics,
// and the rotary table (cos, sin of n * base^(-2i/128) for every token n, at least 32 rows, and
// pair i < 64), computed on the host in double precision once per plan.
int ensure_prep_workspace(fsa_plan_s* P, int H, int D)
{
    const int64_t nb32 = (P->N + 31) / 32;
    const int64_t hf = static_cast<int64_t>(H) * P->F;
    int rc;
    if ((rc = grow(&P->d_rinv, &P->cap_rinv, P->N)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_kpart, &P->cap_kpart, static_cast<int64_t>(H) * nb32 * 2 * D)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_ks, &P->cap_ks, hf)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_kbar, &P->cap_kbar, hf * D)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_gsync, &P->cap_gsync, int64_t(3))) != FSA_OK) return rc;
    if (P->d_rope == nullptr || P->rope_d != D) {
        cudaFree(P->d_rope);
        P->d_rope = nullptr;
        P->rope_d = 0;
        // at least 32 rows: the kernel builds every angle from row n_first and rows 0..31
        const int64_t rows = std::max<int64_t>(P->N, 32);
        const int half = D / 2;
        std::vector<float2> tab(static_cast<size_t>(rows) * half);
        std::vector<double> theta(half);
        for (int i = 0; i < half; ++i) theta[i] = std::pow(kPrepRopeBase, -2.0 * i / D);
        for (int64_t n = 0; n < rows; ++n)
            for (int i = 0; i < half; ++i) {
                const double a = static_cast<double>(n) * theta[i];
                tab[static_cast<size_t>(n) * half + i] = make_float2(static_cast<float>(std::cos(a)),
                                                                     static_cast<float>(std::sin(a)));
            }
        float2* d = nullptr;
        if (cudaMalloc(reinterpret_cast<void**>(&d), tab.size() * sizeof(float2)) != cudaSuccess) return FSA_ERR_CUDA;
        if (cudaMemcpy(d, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(d);
            return FSA_ERR_CUDA;
        }
        P->d_rope = d;
        P->rope_d = D;
    }
    return FSA_OK;
}

// Device copies of a host problem, streams and events for fsa_forward_host.
int ensure_host_pipeline(fsa_plan_s* P, int H, int D, int chunks)
{
    const int64_t in = static_cast<int64_t>(H) * P->N * D;
    const int64_t hn = static_cast<int64_t>(H) * P->N;
    int rc;
    if (P->cap_in < in) {
        cudaFree(P->d_hq);
        cudaFree(P->d_hk);
        cudaFree(P->d_hv);
        P->d_hq = P->d_hk = P->d_hv = nullptr;
        P->cap_in = 0;
        if (cudaMalloc(reinterpret_cast<void**>(&P->d_hq), in * 2) != cudaSuccess ||
            cudaMalloc(reinterpret_cast<void**>(&P->d_hk), in * 2) != cudaSuccess ||
            cudaMalloc(reinterpret_cast<void**>(&P->d_hv), in * 2) != cudaSuccess)
            return FSA_ERR_CUDA;
        P->cap_in = in;
    }
    if ((rc = grow(&P->d_hout, &P->cap_out, in)) != FSA_OK) return rc;
    if ((rc = grow(&P->d_hlse, &P->cap_lse, hn)) != FSA_OK) return rc;
    for (cudaStream_t* s : {&P->s_in, &P->s_comp, &P->s_out})
        if (!*s && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) != cudaSuccess) return FSA_ERR_CUDA;
    while (static_cast<int>(P->ev.size()) < 2 * chunks + 1) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return FSA_ERR_CUDA;
        P->ev.push_back(e);
    }
    return FSA_OK;
}

}  // namespace

int fsa::plan_view(const fsa_plan_s* P, PlanView* out)
{
    if (!P || !out) return FSA_ERR_INVALID_ARG;
    out->F = P->F;
    out->T = P->T;
    out->N = P->N;
    out->tau = P->tau;
    out->center_keys = P->center_keys;
    out->runs = P->runs.data();
    return FSA_OK;
}

extern "C" {

int fsa_last_cuda_error(void)
{
    const int e = g_last_cuda_error;
    g_last_cuda_error = 0;
    return e;
}

const char* fsa_status_string(int status)
{
    switch (status) {
        case FSA_OK: return "ok";
        case FSA_ERR_INVALID_ARG: return "invalid argument";
        case FSA_ERR_UNSUPPORTED: return "unsupported";
        case FSA_ERR_CUDA: return "cuda error";
        case FSA_ERR_TIMEOUT: return "device wait timed out";
        case FSA_ERR_SCRATCH_LIMIT: return "problem too large for the fixed no-allocation scratch";
        default: return "unknown status";
    }
}

int fsa_plan(int F, int T, int w, int ref, int block, fsa_plan_t* out)
{
    if (!out) return FSA_ERR_INVALID_ARG;
    if (F < 1 || T < 16 || w < 0 || ref < 0 || ref >= F) return FSA_ERR_INVALID_ARG;
    if (block < 16 || block % 16 != 0 || T % block != 0) return FSA_ERR_INVALID_ARG;
    const int64_t N = static_cast<int64_t>(F) * T;
    if (N >= (int64_t(1) << 31)) return FSA_ERR_INVALID_ARG;
    fsa_plan_s* P = new (std::nothrow) fsa_plan_s();
    if (!P) return FSA_ERR_INVALID_ARG;
    P->F = F;
    P->T = T;
    P->w = w;
    P->ref = ref;
    P->block = block;
    P->N = N;

    // Key frames of every query frame: the window [f-w, f+w] clipped to [0, F) plus the
    // reference frame, each counted once, ascending.
    auto key_frames = [&](int f) {
        std::vector<int> g;
        for (int x = 0; x < F; ++x)
            if (std::abs(f - x) <= w || x == ref) g.push_back(x);
        return g;
    };

    // Block CSR: blocks never straddle a frame because block divides T.
    const int bpf = T / block;  // blocks per frame
    const int64_t nb = N / block;
    int64_t nnz = 0;
    for (int f = 0; f < F; ++f) nnz += static_cast<int64_t>(key_frames(f).size()) * bpf * bpf;
    if (nnz >= (int64_t(1) << 31)) {
        delete P;
        return FSA_ERR_INVALID_ARG;
    }
    try {
        P->row_ptr.resize(static_cast<size_t>(nb + 1));
        P->col_idx.reserve(static_cast<size_t>(nnz));
        P->row_ptr[0] = 0;
        for (int64_t qb = 0; qb < nb; ++qb) {
            const int f = static_cast<int>(qb / bpf);
            for (int g : key_frames(f))
                for (int b = 0; b < bpf; ++b) P->col_idx.push_back(g * bpf + b);
            P->row_ptr[qb + 1] = static_cast<int32_t>(P->col_idx.size());
        }

        // Key runs per query frame, read off the CSR row of the frame's first block:
        // consecutive key blocks merge into one contiguous run of tokens.
        P->runs.assign(static_cast<size_t>(F) * kRunStride, 0);
        for (int f = 0; f < F; ++f) {
            const int64_t qb = static_cast<int64_t>(f) * bpf;
            int32_t* R = &P->runs[static_cast<size_t>(f) * kRunStride];
            int n = 0;
            int64_t prev = -2;
            for (int32_t e = P->row_ptr[qb]; e < P->row_ptr[qb + 1]; ++e) {
                const int64_t kb = P->col_idx[e];
                if (kb == prev + 1) {
                    R[2 * n] += block;  // extend the current run
                } else {
                    if (n == kMaxRuns) {
                        delete P;
                        return FSA_ERR_UNSUPPORTED;
                    }
                    R[1 + 2 * n] = static_cast<int32_t>(kb * block);
                    R[2 + 2 * n] = block;
                    ++n;
                }
                prev = kb;
            }
            R[0] = n;
        }

    } catch (...) {
        delete P;
        return FSA_ERR_INVALID_ARG;
    }
    *out = P;
    return FSA_OK;
}

void fsa_plan_destroy(fsa_plan_t plan)
{
    if (!plan) return;
    if (plan->device != -1) {
        int cur = -1;
        cudaGetDevice(&cur);
        cudaSetDevice(plan->device);
        cudaDeviceSynchronize();
        cudaFree(plan->d_runs);
        cudaFree(plan->d_qnorm);
        cudaFree(plan->d_bound);
        cudaFree(plan->d_kmax);
        cudaFree(plan->d_ksum);
        cudaFree(plan->d_gmax);
        cudaFree(plan->d_psum);
        cudaFree(plan->d_pmax);
        cudaFree(plan->d_tickets);
        cudaFree(plan->d_htickets);
        cudaFree(plan->d_mu);
        cudaFree(plan->d_rinv);
        cudaFree(plan->d_kpart);
        cudaFree(plan->d_ks);
        cudaFree(plan->d_kbar);
        cudaFree(plan->d_rope);
        cudaFree(plan->d_gsync);
        cudaFree(plan->d_elig);
        cudaFree(plan->d_hq);
        cudaFree(plan->d_hk);
        cudaFree(plan->d_hv);
        cudaFree(plan->d_hout);
        cudaFree(plan->d_hlse);
        cudaFree(plan->d_mask_win);
        cudaFree(plan->d_mask_ref);
        cudaFree(plan->d_out2);
        cudaFree(plan->d_lse2);
        for (cudaStream_t s : {plan->s_in, plan->s_comp, plan->s_out})
            if (s) cudaStreamDestroy(s);
        for (cudaEvent_t e : plan->ev) cudaEventDestroy(e);
        if (cur >= 0) cudaSetDevice(cur);
    }
    delete plan;
}

int fsa_plan_export(fsa_plan_t plan, int32_t* row_ptr, int32_t* col_idx, int64_t* nnz)
{
    if (!plan) return FSA_ERR_INVALID_ARG;
    if (nnz) *nnz = static_cast<int64_t>(plan->col_idx.size());
    if (row_ptr) std::memcpy(row_ptr, plan->row_ptr.data(), plan->row_ptr.size() * sizeof(int32_t));
    if (col_idx && !plan->col_idx.empty())
        std::memcpy(col_idx, plan->col_idx.data(), plan->col_idx.size() * sizeof(int32_t));
    return FSA_OK;
}

int fsa_plan_set_tau(fsa_plan_t plan, float tau)
{
    if (!plan || !(tau > 0.0f)) return FSA_ERR_INVALID_ARG;
    plan->tau = tau;
    return FSA_OK;
}

int fsa_plan_set_center_keys(fsa_plan_t plan, int on)
{
    if (!plan || (on != 0 && on != 1)) return FSA_ERR_INVALID_ARG;
    plan->center_keys = on;
    return FSA_OK;
}

int fsa_plan_set_key_tile(fsa_plan_t plan, int key_tile)
{
    if (!plan) return FSA_ERR_INVALID_ARG;
    if (key_tile != 0 && (key_tile < 16 || key_tile > 128 || key_tile % 16 != 0))
        return FSA_ERR_INVALID_ARG;
    plan->key_tile = key_tile;
    return FSA_OK;
}

int fsa_norms(const uint16_t* q, const uint16_t* k, int H, int D, fsa_plan_t plan, float* qnorm, float* kmax,
              float* bound, uint8_t* eligible, void* stream)
{
    int rc = check_shape(plan, H, D);
    if (rc != FSA_OK) return rc;
    if (H == 0) return FSA_OK;
    if (!q || !k || !aligned16(q) || !aligned16(k)) return FSA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(plan->mu);
    if ((rc = ensure_device(plan)) != FSA_OK) return rc;
    if ((rc = ensure_workspace(plan, H, D)) != FSA_OK) return rc;
    return run_norms(plan, q, k, H, D, qnorm, kmax, bound, eligible, static_cast<cudaStream_t>(stream));
}

int fsa_prep(const uint16_t* x, const uint16_t* w, int d_model, int H, int D, fsa_plan_t plan, uint16_t* q,
             uint16_t* k, uint16_t* v, float* qnorm, float* kmax, float* bound, uint8_t* eligible,
             fsa_stats_t* dev_stats, void* stream)
{
    int rc = check_shape(plan, H, D);
    if (rc != FSA_OK) return rc;
    if ((D != 64 && D != 128) || (H * D) % 256 != 0 || plan->center_keys) return FSA_ERR_UNSUPPORTED;
    if (d_model <= 0 || d_model % 64 != 0) return FSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(3) * H * D * d_model >= (int64_t(1) << 40)) return FSA_ERR_INVALID_ARG;
    if (H == 0) return FSA_OK;
    if (!x || !w || !q || !k || !v) return FSA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return FSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(plan->mu);
    if ((rc = ensure_device(plan)) != FSA_OK) return rc;
    if ((rc = ensure_workspace(plan, H, D)) != FSA_OK) return rc;
    if ((rc = ensure_prep_workspace(plan, H, D)) != FSA_OK) return rc;
    if (dev_stats && (rc = cuda_status(cudaMemsetAsync(dev_stats, 0, sizeof(fsa_stats_t), st))) != FSA_OK) return rc;
    float* km = kmax ? kmax : plan->d_kmax;
    if ((rc = cuda_status(cudaMemsetAsync(km, 0, static_cast<size_t>(H) * plan->F * sizeof(float), st))) != FSA_OK)
        return rc;
    CUtensorMap mx, mw;
    if ((rc = make_tensor_map(&mx, x, plan->N, d_model, 256)) != FSA_OK) return rc;
    if ((rc = make_tensor_map(&mw, w, static_cast<int64_t>(3) * H * D, d_model, 256)) != FSA_OK) return rc;
    fsa::PrepLaunch L;
    L.tmX = &mx;
    L.tmW = &mw;
    L.x = x;
    L.eps = kPrepEps;
    L.D = D;
    L.sms = plan->sms;
    L.stream = st;
    fsa::PrepParams& p = L.params;
    p.N = static_cast<int>(plan->N);
    p.dm = d_model;
    p.H = H;
    p.T = plan->T;
    p.F = plan->F;
    p.m_tiles = static_cast<int>((plan->N + 255) / 256);
    p.tiles_kv = p.m_tiles * (H * D / 128);
    p.rinv = plan->d_rinv;
    p.rope = plan->d_rope;
    p.q = q;
    p.k = k;
    p.v = v;
    p.qnorm = qnorm;
    p.bound = bound ? bound : plan->d_bound;
    p.kmax = reinterpret_cast<unsigned*>(km);
    p.kpart = plan->d_kpart;
    p.ks = plan->d_ks;
    p.kbar = plan->d_kbar;
    p.gmax = plan->d_gmax;
    p.ksum = plan->d_ksum;
    p.runs = plan->d_runs;
    p.gsync = plan->d_gsync;
    p.scale = 1.0f / std::sqrt(static_cast<float>(D));
    p.stats = dev_stats;
    p.wait_limit = kDefaultWaitLimit;
    if (fsa::launch_prep(L) != 0) return FSA_ERR_CUDA;
    return fsa::launch_eligibility(plan->d_gmax, plan->tau, eligible ? eligible : plan->d_elig, H, st) == 0
               ? FSA_OK
               : FSA_ERR_CUDA;
}

int fsa_forward_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse, int H, int D,
                   fsa_plan_t plan, int mode, const float* bound, const uint8_t* eligible, float* rowmax,
                   fsa_stats_t* dev_stats, void* stream)
{
    int rc = check_shape(plan, H, D);
    if (rc != FSA_OK) return rc;
    if (mode != FSA_MODE_NORM_BOUND && mode != FSA_MODE_ONLINE_MAX) return FSA_ERR_INVALID_ARG;
    if ((bound == nullptr) != (eligible == nullptr)) return FSA_ERR_INVALID_ARG;
    if (H == 0) return FSA_OK;  // empty problem: nothing to read or write
    if (!q || !k || !v || !out || !lse) return FSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FSA_ERR_INVALID_ARG;
    const int NK = plan->key_tile ? plan->key_tile : fsa::kMaxKeyTile;
    if (NK > fsa::kMaxKeyTile) return FSA_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(plan->mu);
    if ((rc = ensure_device(plan)) != FSA_OK) return rc;
    if (dev_stats && (rc = cuda_status(cudaMemsetAsync(dev_stats, 0, sizeof(fsa_stats_t), st))) != FSA_OK) return rc;
    return forward_locked(plan, q, k, v, out, lse, H, D, NK, mode, bound, eligible, rowmax, dev_stats, st);
}

int fsa_forward_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse, int H,
                       int D, fsa_plan_t plan, int block, fsa_stats_t* dev_stats, void* stream)
{
    int rc = check_shape(plan, H, D);
    if (rc != FSA_OK) return rc;
    if (block < 128 || block > 1024 || block % 128 != 0) return FSA_ERR_INVALID_ARG;
    if (H == 0) return FSA_OK;
    if (!q || !k || !v || !out || !lse) return FSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FSA_ERR_INVALID_ARG;
    // the padded key range of the last query block must stay inside int32 token indices
    if ((plan->N + block) * static_cast<int64_t>(H) >= (int64_t(1) << 31)) return FSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(plan->mu);
    if ((rc = ensure_device(plan)) != FSA_OK) return rc;
    if (plan->mask_block != block) {
        std::vector<int32_t> win, refp;
        masked_items(plan, block, win, refp);
        cudaFree(plan->d_mask_win);
        cudaFree(plan->d_mask_ref);
        plan->d_mask_win = plan->d_mask_ref = nullptr;
        plan->mask_block = 0;
        if ((rc = upload(&plan->d_mask_win, win)) != FSA_OK || (rc = upload(&plan->d_mask_ref, refp)) != FSA_OK)
            return rc;
        plan->mask_n_win = static_cast<int>(win.size() / kRunStride);
        plan->mask_n_ref = static_cast<int>(refp.size() / kRunStride);
        plan->mask_block = block;
    }
    const int64_t rows = static_cast<int64_t>(H) * plan->N;
    if (plan->mask_n_ref > 0) {
        if ((rc = grow(&plan->d_out2, &plan->cap_out2, rows * D)) != FSA_OK) return rc;
        if ((rc = grow(&plan->d_lse2, &plan->cap_lse2, rows)) != FSA_OK) return rc;
    }
    if (dev_stats && (rc = cuda_status(cudaMemsetAsync(dev_stats, 0, sizeof(fsa_stats_t), st))) != FSA_OK) return rc;
    CUtensorMap mq, mk, mv;
    if ((rc = make_tensor_map(&mq, q, rows, D, 128)) != FSA_OK) return rc;
    if ((rc = make_tensor_map(&mk, k, rows, D, fsa::kMaxKeyTile)) != FSA_OK) return rc;
    if ((rc = make_tensor_map(&mv, v, rows, D, fsa::kMaxKeyTile)) != FSA_OK) return rc;
    for (int pass = 0; pass < 2; ++pass) {
        const int n_items = pass == 0 ? plan->mask_n_win : plan->mask_n_ref;
        if (n_items == 0) continue;
        fsa::AttnLaunch L;
        L.D = D;
        L.H = H;
        L.masked = true;
        L.sms = plan->sms;
        L.tmQ = &mq;
        L.tmK = &mk;
        L.tmV = &mv;
        L.stream = st;
        fsa::AttnParams& a = L.params;
        a.runs = pass == 0 ? plan->d_mask_win : plan->d_mask_ref;
        a.n_tab = n_items;
        a.F = plan->F;
        a.T = plan->T;
        a.N = static_cast<int>(plan->N);
        a.n_qt = 1;
        a.per_head = n_items;
        a.total = H * n_items;
        a.NK = fsa::kMaxKeyTile;
        a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
        a.mode = FSA_MODE_ONLINE_MAX;
        a.bound = nullptr;
        a.eligible = nullptr;
        a.out = pass == 0 ? out : plan->d_out2;
        a.lse = pass == 0 ? lse : plan->d_lse2;
        a.rowmax = nullptr;
        a.stats = dev_stats;
        a.wait_limit = kDefaultWaitLimit;
        a.mask_w = plan->w;
        a.mask_ref = plan->ref;
        a.mask_pass = pass;
        rc = fsa::launch_attention(L);
        if (rc != 0) return rc == -2 ? FSA_ERR_UNSUPPORTED : FSA_ERR_CUDA;
    }
    if (plan->mask_n_ref > 0 &&
        fsa::launch_masked_merge(out, lse, plan->d_out2, plan->d_lse2, H, static_cast<int>(plan->N), plan->T,
                                 plan->F, plan->w, plan->ref, D, st) != 0)
        return FSA_ERR_CUDA;
    return FSA_OK;
}

int fsa_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse, int H, int D,
                fsa_plan_t plan, int mode, void* stream)
{
    return fsa_forward_ex(q, k, v, out, lse, H, D, plan, mode, nullptr, nullptr, nullptr, nullptr, stream);
}

int fsa_forward_host(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* out, float* lse, int H, int D,
                     fsa_plan_t plan, int mode, int heads_per_chunk, void* stream)
{
    int rc = check_shape(plan, H, D);
    if (rc != FSA_OK) return rc;
    if (mode != FSA_MODE_NORM_BOUND && mode != FSA_MODE_ONLINE_MAX) return FSA_ERR_INVALID_ARG;
    if (heads_per_chunk < 0) return FSA_ERR_INVALID_ARG;
    if (H == 0) return FSA_OK;
    if (!q || !k || !v || !out || !lse) return FSA_ERR_INVALID_ARG;
    const int NK = plan->key_tile ? plan->key_tile : fsa::kMaxKeyTile;
    if (NK > fsa::kMaxKeyTile) return FSA_ERR_UNSUPPORTED;
    const int hc = heads_per_chunk ? std::min(heads_per_chunk, H) : std::max(1, (H + 7) / 8);
    const int chunks = (H + hc - 1) / hc;
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(plan->mu);
    if ((rc = ensure_device(plan)) != FSA_OK) return rc;
    if ((rc = ensure_host_pipeline(plan, H, D, chunks)) != FSA_OK) return rc;
    if (mode == FSA_MODE_NORM_BOUND && (rc = ensure_workspace(plan, H, D)) != FSA_OK) return rc;
    fsa_plan_s* P = plan;
    const int64_t per_head = P->N * D;  // elements of one head's q, k, v or out
    cudaEvent_t start = P->ev[2 * chunks];
    // the pipeline starts after the work already on the caller's stream
    if (cudaEventRecord(start, caller) != cudaSuccess || cudaStreamWaitEvent(P->s_in, start, 0) != cudaSuccess)
        return FSA_ERR_CUDA;
    for (int c = 0; c < chunks; ++c) {
        const int h0 = c * hc;
        const int nh = std::min(hc, H - h0);
        const int64_t off = h0 * per_head;
        const size_t in_bytes = static_cast<size_t>(nh) * per_head * 2;
        cudaEvent_t landed = P->ev[2 * c], done = P->ev[2 * c + 1];
        if (cudaMemcpyAsync(P->d_hq + off, q + off, in_bytes, cudaMemcpyHostToDevice, P->s_in) != cudaSuccess ||
            cudaMemcpyAsync(P->d_hk + off, k + off, in_bytes, cudaMemcpyHostToDevice, P->s_in) != cudaSuccess ||
            cudaMemcpyAsync(P->d_hv + off, v + off, in_bytes, cudaMemcpyHostToDevice, P->s_in) != cudaSuccess ||
            cudaEventRecord(landed, P->s_in) != cudaSuccess || cudaStreamWaitEvent(P->s_comp, landed, 0) != cudaSuccess)
            return FSA_ERR_CUDA;
        const float* bnd = nullptr;
        const uint8_t* elg = nullptr;
        if (mode == FSA_MODE_NORM_BOUND) {
            float* b = P->d_bound + h0 * P->N;
            uint8_t* e = P->d_elig + h0;
            if ((rc = run_norms(P, P->d_hq + off, P->d_hk + off, nh, D, nullptr, nullptr, b, e, P->s_comp)) != FSA_OK)
                return rc;
            bnd = b;
            elg = e;
        }
        if ((rc = forward_locked(P, P->d_hq + off, P->d_hk + off, P->d_hv + off, P->d_hout + off,
                                 P->d_hlse + h0 * P->N, nh, D, NK, mode, bnd, elg, nullptr, nullptr, P->s_comp)) !=
            FSA_OK)
            return rc;
        if (cudaEventRecord(done, P->s_comp) != cudaSuccess || cudaStreamWaitEvent(P->s_out, done, 0) != cudaSuccess ||
            cudaMemcpyAsync(out + off, P->d_hout + off, static_cast<size_t>(nh) * per_head * 4,
                            cudaMemcpyDeviceToHost, P->s_out) != cudaSuccess ||
            cudaMemcpyAsync(lse + h0 * P->N, P->d_hlse + h0 * P->N, static_cast<size_t>(nh) * P->N * 4,
                            cudaMemcpyDeviceToHost, P->s_out) != cudaSuccess)
            return FSA_ERR_CUDA;
    }
    // the caller's stream resumes once the last results are on the host
    if (cudaEventRecord(start, P->s_out) != cudaSuccess || cudaStreamWaitEvent(caller, start, 0) != cudaSuccess)
        return FSA_ERR_CUDA;
    return FSA_OK;
}

int fsa_selftest_wait_timeout(long long limit_cycles, int32_t* status, void* stream)
{
    if (!status || limit_cycles <= 0) return FSA_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc != FSA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* d = nullptr;
    if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return FSA_ERR_CUDA;
    rc = cuda_status(cudaMemsetAsync(d, 0, sizeof(int), st));
    if (rc == FSA_OK && fsa::launch_selftest_wait(limit_cycles, d, st) != 0) rc = FSA_ERR_CUDA;
    if (rc == FSA_OK) rc = cuda_status(cudaMemcpyAsync(status, d, sizeof(int), cudaMemcpyDeviceToHost, st));
    if (rc == FSA_OK) rc = cuda_status(cudaStreamSynchronize(st));
    cudaFree(d);
    return rc;
}

int fsa_selftest_grid_timeout(long long limit_cycles, int ctas, int missing, int32_t* result, void* stream)
{
    if (!result || limit_cycles <= 0 || ctas < 1 || (missing != 0 && missing != 1)) return FSA_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc != FSA_OK) return rc;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FSA_ERR_CUDA;
    if (ctas > sms) return FSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* d = nullptr;
    if (cudaMalloc(&d, 8 * sizeof(int)) != cudaSuccess) return FSA_ERR_CUDA;
    rc = cuda_status(cudaMemsetAsync(d, 0, 8 * sizeof(int), st));
    if (rc == FSA_OK &&
        fsa::launch_selftest_grid(limit_cycles, ctas, missing, reinterpret_cast<unsigned*>(d + 4), d, st) != 0)
        rc = FSA_ERR_CUDA;
    if (rc == FSA_OK) rc = cuda_status(cudaMemcpyAsync(result, d, 4 * sizeof(int), cudaMemcpyDeviceToHost, st));
    if (rc == FSA_OK) rc = cuda_status(cudaStreamSynchronize(st));
    cudaFree(d);
    return rc;
}

}  // extern "C"
