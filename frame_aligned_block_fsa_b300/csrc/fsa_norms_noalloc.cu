// fsa_norms_noalloc.cu -- fsa_norms for callers that must not allocate device memory.
//
// fsa_norms keeps its scratch (per-frame key sums, per-head gap maxima) in a plan-owned
// workspace that it grows with cudaMalloc.  Some callers cannot allow that: engines that own the
// whole device memory budget and hand every buffer out themselves, and loops that cannot take
// the device synchronisation cudaMalloc/cudaFree imply.  fsa_norms_noalloc runs the same kernels
// with that scratch in one file-scope device array of fixed size instead, and reads no host
// buffer: the plan's key runs reach the array as kernel arguments of a small fill kernel.
//
// The array is part of the library image: every GPU that loads the library holds it
// (kNoAllocScratchBytes) until the process exits.  Host code cannot use the array's name as a
// device address (on the host it names a host-side stand-in), so the first call on each device
// looks the address up with cudaGetSymbolAddress, with that device current, and caches it with
// the CUDA context it belongs to; a call in another context (after a device reset, say) looks it
// up again.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fsa.h"
#include "fsa_internal.h"

namespace fsa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB

static __device__ __align__(256) unsigned char g_norms_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// Words of the plan's key runs passed by value to one fill launch (within the 4 KB of kernel
// arguments).
constexpr int kFillWords = 960;
struct FillArgs {
    int32_t w[kFillWords];
};

__global__ void fill_runs_kernel(int32_t* dst, int count, const FillArgs a)
{
    for (int i = threadIdx.x; i < count; i += blockDim.x) dst[i] = a.w[i];
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, reached through the runtime (the library links no libcuda).
CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array on the current device (looked up once per device).
int scratch_on_current_device(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FSA_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return FSA_ERR_CUDA;
    if (major != 10 || minor != 3) return FSA_ERR_UNSUPPORTED;
    // make sure the device's context exists and is current, then read it
    if (cudaFree(nullptr) != cudaSuccess) return FSA_ERR_CUDA;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_norms_scratch) != cudaSuccess || p == nullptr) return FSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return FSA_OK;
}

}  // namespace
}  // namespace fsa

extern "C" int fsa_norms_noalloc(const uint16_t* q, const uint16_t* k, int H, int D, fsa_plan_t plan,
                                 float* qnorm, float* kmax, float* bound, uint8_t* eligible, void* stream)
{
    fsa::PlanView pv;
    if (fsa::plan_view(plan, &pv) != FSA_OK || H < 0) return FSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(H) * pv.N >= (int64_t(1) << 31)) return FSA_ERR_INVALID_ARG;
    if (H == 0) return FSA_OK;
    if (!q || !k || !kmax || !bound || !eligible) return FSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k)) & 15u) return FSA_ERR_INVALID_ARG;

    // scratch layout: per-frame tickets and two per-head tickets | key runs of every query
    // frame | per-frame key sums | per-chunk key sums | per-chunk max key norms | per-head gap
    // maxima | per-head key means (used with centred keys)
    const size_t hf = static_cast<size_t>(H) * pv.F;
    const size_t chunks = static_cast<size_t>(fsa::norms_key_chunks(pv.T));
    const size_t tickets_bytes = (hf + 2 * static_cast<size_t>(H)) * sizeof(unsigned);
    const size_t runs_bytes = static_cast<size_t>(pv.F) * fsa::kRunStride * sizeof(int32_t);
    const size_t off_runs = fsa::round256(tickets_bytes);
    const size_t off_ksum = off_runs + fsa::round256(runs_bytes);
    const size_t off_psum = off_ksum + fsa::round256(hf * D * sizeof(float));
    const size_t off_pmax = off_psum + fsa::round256(hf * chunks * D * sizeof(float));
    const size_t off_gmax = off_pmax + fsa::round256(hf * chunks * sizeof(float));
    const size_t off_mu = off_gmax + fsa::round256(static_cast<size_t>(H) * sizeof(unsigned));
    const size_t total = off_mu + fsa::round256(static_cast<size_t>(H) * D * sizeof(float));
    if (total > fsa::kNoAllocScratchBytes) return FSA_ERR_SCRATCH_LIMIT;

    void* base = nullptr;
    int rc = fsa::scratch_on_current_device(&base);
    if (rc != FSA_OK) return rc;
    unsigned char* s = static_cast<unsigned char*>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The previous call's contents are overwritten: the tickets are zeroed and the runs written
    // here (by value, no host buffer is read on the stream), the key sums are written by the
    // first kernel, and the gap maxima are zeroed by the first kernel before the second
    // max-reduces.
    if (cudaMemsetAsync(s, 0, tickets_bytes, st) != cudaSuccess) return FSA_ERR_CUDA;
    const int words = pv.F * fsa::kRunStride;
    for (int w0 = 0; w0 < words; w0 += fsa::kFillWords) {
        fsa::FillArgs a;
        const int cnt = words - w0 < fsa::kFillWords ? words - w0 : fsa::kFillWords;
        for (int i = 0; i < cnt; ++i) a.w[i] = pv.runs[w0 + i];
        fsa::fill_runs_kernel<<<1, 256, 0, st>>>(reinterpret_cast<int32_t*>(s + off_runs) + w0, cnt, a);
        if (cudaGetLastError() != cudaSuccess) return FSA_ERR_CUDA;
    }

    fsa::NormsLaunch L;
    L.q = q;
    L.k = k;
    L.H = H;
    L.D = D;
    L.F = pv.F;
    L.T = pv.T;
    L.N = static_cast<int>(pv.N);
    L.runs = reinterpret_cast<const int32_t*>(s + off_runs);
    L.scale = 1.0f / sqrtf(static_cast<float>(D));
    L.tau = pv.tau;
    L.qnorm = qnorm;
    L.kmax = kmax;
    L.ksum = reinterpret_cast<float*>(s + off_ksum);
    L.part_sum = reinterpret_cast<float*>(s + off_psum);
    L.part_max = reinterpret_cast<float*>(s + off_pmax);
    L.tickets = reinterpret_cast<unsigned*>(s);
    L.bound = bound;
    L.gmax = reinterpret_cast<unsigned*>(s + off_gmax);
    L.eligible = eligible;
    L.center = pv.center_keys;
    L.mu = reinterpret_cast<float*>(s + off_mu);
    L.htickets = reinterpret_cast<unsigned*>(s) + hf;
    L.stream = st;
    rc = fsa::launch_norms(L);
    return rc == 0 ? FSA_OK : (rc == -2 ? FSA_ERR_UNSUPPORTED : FSA_ERR_CUDA);
}
