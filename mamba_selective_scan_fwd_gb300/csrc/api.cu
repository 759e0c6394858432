// C ABI of the selective scan (declared in include/ss.h).
//
// Validation follows the checks of the baracuda-kernels `selective_scan.rs`
// plans (`SelectiveScanPlan::select`, `can_implement`, `run` and the
// backward's `run`): negative extents and missing or inconsistent optional
// tensors are invalid problems, unsupported dtypes / state sizes are
// unsupported, a short workspace is reported before any launch.  Everything
// is checked before the first CUDA call; on error nothing is written.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ss.h"
#include "common.cuh"
#include "kernels.h"

using namespace ss;

namespace {

// ---------------------------------------------------------------- device status word
// A kernel that gives up waiting for one of its copies leaves a code here
// (kDevWaitTimeout) and returns; ss_device_status reads and clears it.
static __device__ int g_status;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
int* g_status_ptr[kMaxDevices] = {};

// Device address of g_status on the current device (looked up once per device).
int status_for_current_device(int** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess || ptr == nullptr) return SS_ERR_CUDA;
        g_status_ptr[dev] = static_cast<int*>(ptr);
    }
    *out = g_status_ptr[dev];
    return SS_OK;
}

// One block that waits on a barrier nothing completes, for at most limit_ns:
// the wait runs out and the block records it like a scan kernel would.
__global__ void k_wait_timeout(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_proxy_async_smem();
        if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(status, kDevWaitTimeout);
    }
}

// ---------------------------------------------------------------- tensor maps
// cuTensorMapEncodeTiled, taken from the driver through the runtime (no link
// against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// 0: TMA staging wherever the problem allows it; 1: asynchronous copies only.
std::atomic<int> g_copies_only{0};

// A [Bsz, L, inner] tensor as a 3-D map {inner, L, Bsz} with boxes of
// {box_x, rows, 1}; rows and channels outside the tensor read as zero.
bool encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType type, int esz, int64_t Bsz, int64_t L,
                int64_t inner, int box_x, int rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)Bsz};
    const cuuint64_t strides[2] = {(cuuint64_t)(inner * esz), (cuuint64_t)(inner * L * esz)};
    const cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether the scan kernels of this problem stage their tiles with TMA: every
// box's row is a whole number of 16-byte units (D and N times the element
// size), the tensors' row strides are multiples of 16 bytes, the strides and
// coordinates fit the map's ranges, and the driver provides the encoder.
bool tma_eligible(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (g_copies_only.load(std::memory_order_relaxed)) return false;
    const int64_t esz = dtype == SS_F32 ? 4 : 2;
    if ((Dch * esz) % 16 != 0 || (N * esz) % 16 != 0 || Dch % 4 != 0) return false;
    if (L >= (1ll << 31) || Bsz >= (1ll << 31) || Dch * L * 4 >= (1ll << 40)) return false;
    return encode_fn() != nullptr;
}

// The maps a forward (rows = steps per tile of the forward) or a backward
// (rows = steps per staging copy: two recompute windows for two-warp blocks,
// one otherwise) loads its tiles through; y0 (f32, the forward's pre-gate
// readout kept for dz) only for the backward.
bool make_maps(TmaMaps& mp, const FwdArgs& f, const void* dy, const float* y0, int rows) {
    const CUtensorMapDataType io = f.dtype == SS_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : f.dtype == SS_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int esz = f.dtype == SS_F32 ? 4 : 2;
    const int CH = (int)channels_per_block((int)f.N);
    bool ok = encode_map(&mp.m[kMapDelta], f.delta, io, esz, f.Bsz, f.L, f.Dch, CH, rows) &&
              encode_map(&mp.m[kMapU], f.u, io, esz, f.Bsz, f.L, f.Dch, CH, rows) &&
              encode_map(&mp.m[kMapB], f.B, io, esz, f.Bsz, f.L, f.N, (int)f.N, rows) &&
              encode_map(&mp.m[kMapC], f.C, io, esz, f.Bsz, f.L, f.N, (int)f.N, rows);
    if (ok && f.z) ok = encode_map(&mp.m[kMapZ], f.z, io, esz, f.Bsz, f.L, f.Dch, CH, rows);
    if (ok && dy) ok = encode_map(&mp.m[kMapDy], dy, io, esz, f.Bsz, f.L, f.Dch, CH, rows);
    if (ok && y0) ok = encode_map(&mp.m[kMapY0], y0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, f.Bsz, f.L, f.Dch, CH, rows);
    return ok;
}

bool n_supported(int64_t N) { return N == 1 || N == 2 || N == 4 || N == 8 || N == 16 || N == 32; }

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (Bsz < 0 || L < 0 || Dch < 0 || N < 0) return SS_ERR_INVALID_PROBLEM;
    if (dtype != SS_F32 && dtype != SS_F16 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
    if (!n_supported(N)) return SS_ERR_UNSUPPORTED;
    // index products stay far inside int64; grid sizes stay inside 2^31 - 1 blocks
    if (Bsz > (1ll << 20) || L > (1ll << 31) || Dch > (1ll << 24)) return SS_ERR_UNSUPPORTED;
    if (Bsz * L > (1ll << 40) || Bsz * L * Dch > (1ll << 46)) return SS_ERR_UNSUPPORTED;
    return SS_OK;
}

// ss_profile_events state: the caller's events and the next one to record,
// per host thread (a list set by one thread applies to that thread's calls).
constexpr int kMaxProfEvents = 16;
thread_local cudaEvent_t g_prof_ev[kMaxProfEvents];
thread_local int g_prof_n = 0;
thread_local int g_prof_next = 0;

// Forward with optional restart-state output (save == false: plain forward),
// initial state h0 (nullable) and the A_log form.
int fwd_impl(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
             const void* z, const float* delta_bias, const float* h0, int softplus, int a_is_log, void* y,
             float* last_state, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, bool save, void* saved,
             size_t saved_bytes, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    if (!empty && (!u || !delta || !A || !B || !C || !y)) return SS_ERR_INVALID_PROBLEM;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, h0, y, last_state, saved, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SS_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (empty) {
        // no step: the state stays the initial one
        if (last_state && Bsz > 0 && Dch > 0 && N > 0) {
            const size_t bytes = (size_t)Bsz * Dch * N * sizeof(float);
            const cudaError_t e = h0 ? cudaMemcpyAsync(last_state, h0, bytes, cudaMemcpyDeviceToDevice, st)
                                     : cudaMemsetAsync(last_state, 0, bytes, st);
            if (e != cudaSuccess) return SS_ERR_CUDA;
        }
        return SS_OK;
    }
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    if (ceil_div(Dch, 4) * Bsz * p.Kmax >= (1ll << 31)) return SS_ERR_UNSUPPORTED;
    if (save) {
        const size_t need_s = ckpt_bytes(p, Bsz, L, Dch, N);
        if (saved == nullptr || saved_bytes < need_s) return SS_ERR_WORKSPACE_TOO_SMALL;
    }
    const size_t need = ss_fwd_workspace_bytes(Bsz, L, Dch, N, dtype);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return SS_ERR_WORKSPACE_TOO_SMALL;
    FwdArgs a;
    a.u = u; a.delta = delta; a.B = B; a.C = C; a.z = z;
    a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.h0 = h0;
    a.y = y; a.last_state = last_state;
    a.Bsz = Bsz; a.L = L; a.Dch = Dch; a.N = N;
    a.softplus = softplus ? 1 : 0;
    a.a_is_log = a_is_log ? 1 : 0;
    a.dtype = dtype;
    a.ws_fsum = static_cast<float*>(workspace);
    a.ws_fsd = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) + fsum_offset_sd(p, N)) : nullptr;
    float* ck = save ? static_cast<float*>(saved) : nullptr;
    a.y0 = save ? reinterpret_cast<float*>(static_cast<char*>(saved) + ckpt_y0_offset(p, Bsz, N)) : nullptr;
    rc = status_for_current_device(&a.status);
    if (rc != SS_OK) return rc;
    TmaMaps maps;
    a.use_tma = tma_eligible(Bsz, L, Dch, N, dtype) && make_maps(maps, a, nullptr, nullptr, kFwdRows) ? 1 : 0;
    return launch_fwd(a, p, st, kModeY, ck, maps) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// Backward; with from_saved the restart states come from ss_fwd_save /
// ss_fwd_ex.  h0 / dlast (nullable): initial state and incoming gradient of
// last_state; dh0 (given iff h0): gradient of the initial state.
int bwd_impl(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
             const void* z, const float* delta_bias, const float* h0, int softplus, int a_is_log, const void* dy,
             const float* dlast, float* du, float* ddelta, float* dA, float* dB, float* dC, float* dD, float* dz,
             float* ddelta_bias, float* dh0, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype,
             bool from_saved, const void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
             void* stream) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    if ((D == nullptr) != (dD == nullptr) || (z == nullptr) != (dz == nullptr) ||
        (delta_bias == nullptr) != (ddelta_bias == nullptr) || (h0 == nullptr) != (dh0 == nullptr))
        return SS_ERR_INVALID_PROBLEM;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    if (!empty && (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC))
        return SS_ERR_INVALID_PROBLEM;
    if (empty && Dch > 0 && N > 0 && !dA) return SS_ERR_INVALID_PROBLEM;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, h0, dy, dlast, du, ddelta, dA, dB, dC, dD, dz,
                          ddelta_bias, dh0, saved, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SS_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (empty) {
        // parameter gradients are sums over an empty set: zero
        if (Dch > 0) {
            if (dA && N > 0 && cudaMemsetAsync(dA, 0, (size_t)Dch * N * sizeof(float), st) != cudaSuccess)
                return SS_ERR_CUDA;
            if (dD && cudaMemsetAsync(dD, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess) return SS_ERR_CUDA;
            if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess)
                return SS_ERR_CUDA;
        }
        // L == 0: h0 is last_state, so its gradient is the incoming one
        if (dh0 && Bsz > 0 && Dch > 0 && N > 0) {
            const size_t bytes = (size_t)Bsz * Dch * N * sizeof(float);
            const cudaError_t e = dlast ? cudaMemcpyAsync(dh0, dlast, bytes, cudaMemcpyDeviceToDevice, st)
                                        : cudaMemsetAsync(dh0, 0, bytes, st);
            if (e != cudaSuccess) return SS_ERR_CUDA;
        }
        // Dch == 0 with Bsz, L > 0: dB and dC are sums over no channels
        if (Dch == 0 && Bsz > 0 && L > 0 && N > 0) {
            if (dB && cudaMemsetAsync(dB, 0, (size_t)Bsz * L * N * sizeof(float), st) != cudaSuccess)
                return SS_ERR_CUDA;
            if (dC && cudaMemsetAsync(dC, 0, (size_t)Bsz * L * N * sizeof(float), st) != cudaSuccess)
                return SS_ERR_CUDA;
        }
        return SS_OK;
    }
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    if (ceil_div(Dch, 4) * Bsz * p.Kmax >= (1ll << 31)) return SS_ERR_UNSUPPORTED;
    if (from_saved && (saved == nullptr || saved_bytes < ckpt_bytes(p, Bsz, L, Dch, N)))
        return SS_ERR_WORKSPACE_TOO_SMALL;
    const BwdLayout w = bwd_layout2(p, Bsz, L, Dch, N, from_saved);
    if (workspace_bytes < w.total || workspace == nullptr) return SS_ERR_WORKSPACE_TOO_SMALL;
    char* ws = static_cast<char*>(workspace);
    BwdArgs a;
    a.f.u = u; a.f.delta = delta; a.f.B = B; a.f.C = C; a.f.z = z;
    a.f.A = A; a.f.D = D; a.f.delta_bias = delta_bias;
    a.f.h0 = h0;
    a.f.y = nullptr; a.f.last_state = nullptr;
    a.f.Bsz = Bsz; a.f.L = L; a.f.Dch = Dch; a.f.N = N;
    a.f.softplus = softplus ? 1 : 0;
    a.f.a_is_log = a_is_log ? 1 : 0;
    a.f.dtype = dtype;
    a.f.ws_fsum = reinterpret_cast<float*>(ws + w.fsum);
    a.f.ws_fsd = reinterpret_cast<float*>(ws + w.fsd);
    a.dy = dy;
    a.dlast = dlast;
    a.du = du; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz;
    a.ddelta_bias = ddelta_bias;
    a.dh0 = dh0;
    a.ws_rsum = reinterpret_cast<float*>(ws + w.rsum);
    a.ws_rsd = reinterpret_cast<float*>(ws + w.rsd);
    float* ckpt_out = from_saved ? nullptr : reinterpret_cast<float*>(ws + w.ckpt);
    a.ws_ckpt = from_saved ? static_cast<const float*>(saved) : ckpt_out;
    const char* kept = from_saved ? static_cast<const char*>(saved) : ws + w.ckpt;
    a.y0 = reinterpret_cast<const float*>(kept + ckpt_y0_offset(p, Bsz, N));
    a.f.y0 = from_saved ? nullptr : reinterpret_cast<float*>(ws + w.ckpt + ckpt_y0_offset(p, Bsz, N));
    a.ws_bc = reinterpret_cast<float*>(ws + w.bc);
    a.ws_dA = reinterpret_cast<float*>(ws + w.dA);
    a.ws_dD = reinterpret_cast<float*>(ws + w.dD);
    a.ws_db = reinterpret_cast<float*>(ws + w.db);
    rc = status_for_current_device(&a.f.status);
    if (rc != SS_OK) return rc;
    // the forward passes that store the restart states and the reverse summaries
    // use the forward's 32-step boxes, the main pass its own
    TmaMaps fmaps, bmaps;
    a.f.use_tma = tma_eligible(Bsz, L, Dch, N, dtype) && make_maps(fmaps, a.f, dy, nullptr, kFwdRows) &&
                          make_maps(bmaps, a.f, dy, z ? a.y0 : nullptr, (scan_warps(N) == 2 ? 2 : 1) * kSub)
                      ? 1
                      : 0;
    return launch_bwd(a, p, st, ckpt_out, fmaps, bmaps) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// An entry point's launches between prof_begin and prof_end.
void prof_begin() { g_prof_next = 0; }
int prof_end(cudaStream_t st, int rc) {
    if (rc == SS_OK) ss::prof_mark(st);
    return rc;
}

}  // namespace

namespace ss {
void prof_mark(cudaStream_t st) {
    if (g_prof_next < g_prof_n) cudaEventRecord(g_prof_ev[g_prof_next++], st);
}
}  // namespace ss

extern "C" {

int ss_profile_events(void* const* events, int count) {
    if (count < 0 || count > kMaxProfEvents || (count > 0 && events == nullptr)) return SS_ERR_INVALID_PROBLEM;
    for (int i = 0; i < count; i++)
        if (events[i] == nullptr) return SS_ERR_INVALID_PROBLEM;
    for (int i = 0; i < count; i++) g_prof_ev[i] = static_cast<cudaEvent_t>(events[i]);
    g_prof_n = count;
    g_prof_next = 0;
    return SS_OK;
}

int ss_abi_version(void) { return 7; }

int ss_device_status(void* stream) {
    int* status = nullptr;
    int rc = status_for_current_device(&status);
    if (rc != SS_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return SS_ERR_CUDA;
    if (host & kDevWaitTimeout) return SS_ERR_DEVICE_TIMEOUT;
    return host & kDevMisaligned ? SS_ERR_STAGING_FALLBACK : SS_OK;
}

int ss_selftest_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 0 || limit_ns > (int64_t)kWaitLimitNs) return SS_ERR_INVALID_PROBLEM;
    int* status = nullptr;
    int rc = status_for_current_device(&status);
    if (rc != SS_OK) return rc;
    k_wait_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, (uint64_t)limit_ns);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

int ss_set_copies_only(int enable) { return g_copies_only.exchange(enable ? 1 : 0); }

int ss_staging_uses_tma(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK || Bsz == 0 || L == 0 || Dch == 0) return 0;
    return tma_eligible(Bsz, L, Dch, N, dtype) ? 1 : 0;
}

const char* ss_status_string(int status) {
    switch (status) {
        case SS_OK: return "ok";
        case SS_ERR_INVALID_PROBLEM: return "invalid problem (negative extent, missing pointer or optional-term mismatch)";
        case SS_ERR_UNSUPPORTED: return "unsupported (dtype, state size, size limit or pointer alignment)";
        case SS_ERR_WORKSPACE_TOO_SMALL: return "workspace or saved-state buffer too small (query its *_bytes function)";
        case SS_ERR_CUDA: return "CUDA runtime error";
        case SS_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting for its tile copies (see ss_device_status)";
        case SS_ERR_STAGING_FALLBACK: return "a kernel staged its tiles without TMA (results intact; see ss_device_status)";
        default: return "unknown status";
    }
}

size_t ss_fwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    return fsum_bytes(make_fplan(Bsz, L, Dch, N), N);
}

size_t ss_bwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    return bwd_layout2(p, Bsz, L, Dch, N, false).total;
}

size_t ss_saved_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    return ckpt_bytes(make_fplan(Bsz, L, Dch, N), Bsz, L, Dch, N);
}

size_t ss_bwd_saved_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    return bwd_layout2(p, Bsz, L, Dch, N, true).total;
}

int ss_plan_info(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, int64_t* chunks, int* fwd_kernels,
                 int* bwd_kernels, int* bwd_saved_kernels) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    const FPlan fp = make_fplan(Bsz, L, Dch, N);
    if (chunks) *chunks = empty ? 0 : fp.Kmax;
    // per segment: its main pass, after a summary pass if it is chunked (and in
    // the backward a carry pass after that); the forward (with or without
    // saving) runs the forward passes, the backward from saved states the
    // reverse ones and 2 reductions, the backward the forward checkpoint passes
    // first
    int fscans = 0, rscans = 0;
    for (int i = 0; i < fp.nseg; i++) {
        fscans += 1 + (fp.seg[i].K > 1 ? 1 : 0);
        rscans += 1 + (fp.seg[i].K > 1 ? 2 : 0);
    }
    if (fwd_kernels) *fwd_kernels = empty ? 0 : fscans;
    if (bwd_kernels) *bwd_kernels = empty ? 0 : fscans + rscans + 2;
    if (bwd_saved_kernels) *bwd_saved_kernels = empty ? 0 : rscans + 2;
    return SS_OK;
}

int ss_plan_segments(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, int* nseg, int64_t* units,
                     int64_t* chunks) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    if (Bsz == 0 || L == 0 || Dch == 0) {
        if (nseg) *nseg = 0;
        return SS_OK;
    }
    const FPlan fp = make_fplan(Bsz, L, Dch, N);
    if (nseg) *nseg = fp.nseg;
    for (int i = 0; i < fp.nseg; i++) {
        if (units) units[i] = fp.seg[i].nu;
        if (chunks) chunks[i] = fp.seg[i].K;
    }
    return SS_OK;
}

int ss_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
           const void* z, const float* delta_bias, int softplus, void* y, float* last_state, int64_t Bsz, int64_t L,
           int64_t Dch, int64_t N, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    fwd_impl(u, delta, A, B, C, D, z, delta_bias, nullptr, softplus, 0, y, last_state, Bsz, L, Dch,
                             N, dtype, false, nullptr, 0, workspace, workspace_bytes, stream));
}

int ss_fwd_save(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                const void* z, const float* delta_bias, int softplus, void* y, float* last_state, void* saved,
                size_t saved_bytes, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    fwd_impl(u, delta, A, B, C, D, z, delta_bias, nullptr, softplus, 0, y, last_state, Bsz, L, Dch,
                             N, dtype, true, saved, saved_bytes, workspace, workspace_bytes, stream));
}

int ss_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
           const void* z, const float* delta_bias, int softplus, const void* dy, float* du, float* ddelta, float* dA,
           float* dB, float* dC, float* dD, float* dz, float* ddelta_bias, int64_t Bsz, int64_t L, int64_t Dch,
           int64_t N, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    bwd_impl(u, delta, A, B, C, D, z, delta_bias, nullptr, softplus, 0, dy, nullptr, du, ddelta, dA,
                             dB, dC, dD, dz, ddelta_bias, nullptr, Bsz, L, Dch, N, dtype, false, nullptr, 0, workspace,
                             workspace_bytes, stream));
}

int ss_bwd_saved(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* delta_bias, int softplus, const void* dy, const void* saved,
                 size_t saved_bytes, float* du, float* ddelta, float* dA, float* dB, float* dC, float* dD, float* dz,
                 float* ddelta_bias, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    bwd_impl(u, delta, A, B, C, D, z, delta_bias, nullptr, softplus, 0, dy, nullptr, du, ddelta, dA,
                             dB, dC, dD, dz, ddelta_bias, nullptr, Bsz, L, Dch, N, dtype, true, saved, saved_bytes,
                             workspace, workspace_bytes, stream));
}

int ss_fwd_ex(const ss_fwd_desc* d, void* stream) {
    if (d == nullptr) return SS_ERR_INVALID_PROBLEM;
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    fwd_impl(d->u, d->delta, d->A, d->B, d->C, d->D, d->z, d->delta_bias, d->h0, d->softplus,
                             d->a_is_log, d->y, d->last_state, d->Bsz, d->L, d->Dch, d->N, d->dtype,
                             d->saved != nullptr, d->saved, d->saved_bytes, d->workspace, d->workspace_bytes,
                             stream));
}

int ss_bwd_ex(const ss_bwd_desc* d, void* stream) {
    if (d == nullptr) return SS_ERR_INVALID_PROBLEM;
    prof_begin();
    return prof_end(static_cast<cudaStream_t>(stream),
                    bwd_impl(d->u, d->delta, d->A, d->B, d->C, d->D, d->z, d->delta_bias, d->h0, d->softplus,
                             d->a_is_log, d->dy, d->dlast_state, d->du, d->ddelta, d->dA, d->dB, d->dC, d->dD, d->dz,
                             d->ddelta_bias, d->dh0, d->Bsz, d->L, d->Dch, d->N, d->dtype, d->saved != nullptr,
                             d->saved, d->saved_bytes, d->workspace, d->workspace_bytes, stream));
}

int ss_decode_step(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                   const void* z, const float* delta_bias, int softplus, int a_is_log, float* state, void* y,
                   int64_t Bsz, int64_t Dch, int64_t N, int dtype, void* stream) {
    prof_begin();
    int rc = check_sizes(Bsz, 1, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    if (Bsz == 0 || Dch == 0) return SS_OK;
    if (Bsz * Dch > (1ll << 36)) return SS_ERR_UNSUPPORTED;  // grid of at most 8 threads per (b, d) stays below 2^31 blocks
    if (!u || !delta || !A || !B || !C || !state || !y) return SS_ERR_INVALID_PROBLEM;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, state, y};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SS_ERR_UNSUPPORTED;
    DecodeArgs a;
    a.u = u; a.delta = delta; a.B = B; a.C = C; a.z = z;
    a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.state = state; a.y = y;
    a.Bsz = Bsz; a.Dch = Dch; a.N = N;
    a.softplus = softplus ? 1 : 0;
    a.a_is_log = a_is_log ? 1 : 0;
    a.dtype = dtype;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return prof_end(st, launch_decode(a, st) == cudaSuccess ? SS_OK : SS_ERR_CUDA);
}

}  // extern "C"
