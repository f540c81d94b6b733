// fsa_internal.h -- structures shared by the host API and the kernels (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fsa.h"

namespace fsa {

// Key runs of one query frame: [n_runs, start_0, len_0, start_1, len_1] in tokens of a head;
// every run is a union of whole frames, ascending, disjoint.  A frame's key set is a window
// of consecutive frames plus the reference frame, so it never takes more than two runs.
constexpr int kMaxRuns = 2;
constexpr int kRunStride = 1 + 2 * kMaxRuns;

// Largest key tile of the attention kernel (its two S buffers hold 128 columns each).
constexpr int kMaxKeyTile = 128;

// Work item of the masked block variant (one 128-row query tile of a query block on the padded
// sequence): [first query token, first key token, keys (a multiple of the block size), 0, 0].
// The kernel reads it from the same table slot as a frame's key runs.
constexpr int kMaskItemRow = 0, kMaskItemKey = 1, kMaskItemLen = 2;

struct AttnParams {
    const int32_t* runs;   // frame-aligned: [F][kRunStride] key runs; masked: [per_head][kRunStride] items
    int n_tab;             // entries of `runs` (F, or the masked items per head)
    int F, T, N;           // frames, tokens per frame, tokens per head
    int n_qt;              // 128-row query tiles per frame, ceil(T / 128) (frame-aligned)
    int per_head;          // work items per head: F * n_qt, or the masked items per head
    int total;             // work items, H * per_head
    int NK;                // keys per tile (multiple of 16, at most kMaxKeyTile)
    float scale_log2;      // c * log2(e)
    int mode;              // 0 norm_bound, 1 online_max
    const float* bound;    // [H][N] or null
    const uint8_t* eligible;  // [H] or null
    float* out;            // [H][N][D]
    float* lse;            // [H][N]
    float* rowmax;         // [H][N] or null
    fsa_stats_t* stats;    // or null
    long long wait_limit;  // clock cycles
    // masked block variant: each row's keys are one interval of the sequence, the window of
    // frames [f - w, f + w] clipped to [0, F) (pass 0) or the reference frame when outside that
    // window (pass 1, else no key); keys outside it are masked by predicate
    int mask_w, mask_ref, mask_pass;
};

struct AttnLaunch {
    int D, H;
    bool masked;           // the masked block variant (online softmax only)
    int sms;               // persistent grid: min(sms, work items) CTAs
    const CUtensorMap* tmQ;  // boxes of 128 rows
    const CUtensorMap* tmK;  // boxes of NK rows
    const CUtensorMap* tmV;
    AttnParams params;
    cudaStream_t stream;
};

// Records the code of a failed CUDA call for fsa_last_cuda_error (per host thread).
void note_cuda_error(int code);
// cudaGetLastError after a launch: 0 on success, else -3 with the code recorded.
int launch_status();

int launch_attention(const AttnLaunch& L);
// Merge of the masked variant's two passes, in place on (out, lse): rows whose window leaves out
// the reference frame combine their window-pass result with the reference pass's (out2, lse2).
int launch_masked_merge(float* out, float* lse, const float* out2, const float* lse2, int H, int N, int T, int F,
                        int w, int ref, int D, cudaStream_t stream);
int attn_smem_bytes(int D);
int launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream);
int launch_selftest_grid(long long limit, int ctas, int missing, unsigned* d_counter, int* d_result,
                         cudaStream_t stream);

struct NormsLaunch {
    const uint16_t* q;
    const uint16_t* k;
    int H, D, F, T, N;
    const int32_t* runs;   // device [F][kRunStride]
    float scale;
    float tau;
    float* qnorm;          // [H][N] or null
    float* kmax;           // [H][F]
    float* ksum;           // [H][F][D] workspace
    float* part_sum;       // [H][F][chunks][D] workspace: column sums of a chunk of a frame's keys
    float* part_max;       // [H][F][chunks] workspace: the chunk's max key norm
    unsigned* tickets;     // [H][F] workspace, zero between launches (each launch leaves it zero)
    float* bound;          // [H][N]
    unsigned* gmax;        // [H] workspace
    uint8_t* eligible;     // [H]
    int center;            // 1: key norms about the head's mean key, c <q, mu> added to the bound
    float* mu;             // [H][D] workspace (center only)
    unsigned* htickets;    // [2H] workspace, zero between launches: head key means (center), eligibility
    cudaStream_t stream;
};

int launch_norms(const NormsLaunch& L);
// Chunks of a frame's keys that key_frame_stats reads in separate blocks (1..kMaxKeyChunks).
constexpr int kMaxKeyChunks = 8;
int norms_key_chunks(int T);

int launch_eligibility(const unsigned* gmax, float tau, uint8_t* eligible, int H, cudaStream_t stream);

// The fused preparation of the attention inputs (fsa_prep): D = 64 or 128, H D a multiple of 256.
struct PrepParams {
    int N, dm, H, T, F;
    int m_tiles;             // ceil(N / 256) token-row tiles
    int tiles_kv;            // m_tiles * H D / 128 tiles of K and V columns, before the Q tiles
    float* rinv;             // [N] 1 / rms of each token row
    const float2* rope;      // [max(N, 32)][D/2] (cos, sin) of the rotary angles
    uint16_t* q;             // [H][N][D] outputs
    uint16_t* k;
    uint16_t* v;
    float* qnorm;            // [H][N] or null
    float* bound;            // [H][N]
    unsigned* kmax;          // [H][F] float bits; zero before the K/V launch
    float* kpart;            // [H][ceil(N/32)][2][D] column sums of K per 32-row block and frame
    float* ks;               // [H][F] max key norm over each query frame's key set
    float* kbar;             // [H][F][D] mean key over each query frame's key set
    unsigned* gmax;          // [H] gap maxima (float bits)
    float* ksum;             // [H][F][D] workspace: per-frame key sums
    const int32_t* runs;     // device [F][kRunStride]
    unsigned* gsync;         // [3] grid-barrier counters, zero before the launch
    float scale;             // c = 1/sqrt(D)
    fsa_stats_t* stats;      // or null
    long long wait_limit;    // clock cycles
};

struct PrepLaunch {
    const CUtensorMap* tmX;  // x bf16 [N][dm], boxes 64 x 256
    const CUtensorMap* tmW;  // w bf16 [3 H D][dm], boxes 64 x 256
    const uint16_t* x;
    int D;                   // head dim, 64 or 128
    float eps;
    int sms;                 // persistent grid size (all CTAs co-resident: cooperative launch)
    PrepParams params;
    cudaStream_t stream;
};

int launch_prep(const PrepLaunch& L);
int prep_smem_bytes();

// Read-only view of a plan's host data, for entry points that live outside fsa_api.cpp.
struct PlanView {
    int F, T;
    int64_t N;
    float tau;
    int center_keys;
    const int32_t* runs;  // host [F][kRunStride]
};

int plan_view(const fsa_plan_s* plan, PlanView* out);

}  // namespace fsa
