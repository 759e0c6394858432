// C ABI of the selective scan (declared in include/ss.h).
//
// Validation follows the checks of the baracuda-kernels `selective_scan.rs`
// plans (`SelectiveScanPlan::select`, `can_implement`, `run` and the
// backward's `run`): negative extents and missing or inconsistent optional
// tensors are invalid problems, unsupported dtypes / state sizes are
// unsupported, a short workspace is reported before any launch.  Everything
// is checked before the first CUDA call; on error nothing is written.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ss.h"
#include "common.cuh"
#include "kernels.h"

using namespace ss;

namespace {

bool n_supported(int64_t N) { return N == 1 || N == 2 || N == 4 || N == 8 || N == 16 || N == 32; }

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (Bsz < 0 || L < 0 || Dch < 0 || N < 0) return SS_ERR_INVALID_PROBLEM;
    if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
    if (!n_supported(N)) return SS_ERR_UNSUPPORTED;
    // index products stay far inside int64; grid sizes stay inside 2^31 - 1 blocks
    if (Bsz > (1ll << 20) || L > (1ll << 31) || Dch > (1ll << 24)) return SS_ERR_UNSUPPORTED;
    if (Bsz * L > (1ll << 40) || Bsz * L * Dch > (1ll << 46)) return SS_ERR_UNSUPPORTED;
    return SS_OK;
}

}  // namespace

extern "C" {

int ss_abi_version(void) { return 1; }

const char* ss_status_string(int status) {
    switch (status) {
        case SS_OK: return "ok";
        case SS_ERR_INVALID_PROBLEM: return "invalid problem (negative extent, missing pointer or optional-term mismatch)";
        case SS_ERR_UNSUPPORTED: return "unsupported (dtype, state size, size limit or pointer alignment)";
        case SS_ERR_WORKSPACE_TOO_SMALL: return "workspace too small (query ss_*_workspace_bytes)";
        case SS_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

size_t ss_fwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    if (p.K <= 1) return 0;
    return align_up((size_t)Bsz * Dch * p.K * N * 2 * sizeof(float), 256);
}

size_t ss_bwd_workspace_bytes(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype) {
    if (check_sizes(Bsz, L, Dch, N, dtype) != SS_OK) return 0;
    if (Bsz == 0 || L == 0 || Dch == 0) return 0;
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    return bwd_layout2(p, Bsz, L, Dch, N).total;
}

int ss_plan_info(int64_t Bsz, int64_t L, int64_t Dch, int64_t N, int dtype, int64_t* chunks, int* fwd_kernels,
                 int* bwd_kernels) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    const FPlan fp = make_fplan(Bsz, L, Dch, N);
    if (chunks) *chunks = empty ? 0 : fp.K;
    // forward: [summary if K > 1] + main;
    // backward: [forward summary if K > 1] + checkpoints + [reverse summary if K > 1] + main + 2 reductions
    if (fwd_kernels) *fwd_kernels = empty ? 0 : (fp.K > 1 ? 2 : 1);
    if (bwd_kernels) *bwd_kernels = empty ? 0 : (fp.K > 1 ? 6 : 4);
    return SS_OK;
}

int ss_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
           const void* z, const float* delta_bias, int softplus, void* y, float* last_state, int64_t Bsz, int64_t L,
           int64_t Dch, int64_t N, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    if (!empty && (!u || !delta || !A || !B || !C || !y)) return SS_ERR_INVALID_PROBLEM;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, y, last_state, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SS_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (empty) {
        if (last_state && Bsz > 0 && Dch > 0 && N > 0) {
            if (cudaMemsetAsync(last_state, 0, (size_t)Bsz * Dch * N * sizeof(float), st) != cudaSuccess)
                return SS_ERR_CUDA;
        }
        return SS_OK;
    }
    const FPlan p = make_fplan(Bsz, L, Dch, N);
    if (ceil_div(Dch, 4) * Bsz * p.K >= (1ll << 31)) return SS_ERR_UNSUPPORTED;
    const size_t need = ss_fwd_workspace_bytes(Bsz, L, Dch, N, dtype);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return SS_ERR_WORKSPACE_TOO_SMALL;
    FwdArgs a;
    a.u = u; a.delta = delta; a.B = B; a.C = C; a.z = z;
    a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.y = y; a.last_state = last_state;
    a.Bsz = Bsz; a.L = L; a.Dch = Dch; a.N = N;
    a.softplus = softplus ? 1 : 0;
    a.dtype = dtype;
    a.ws_fsum = static_cast<float*>(workspace);
    return launch_fwd2(a, p, st, kModeY, nullptr) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

int ss_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
           const void* z, const float* delta_bias, int softplus, const void* dy, float* du, float* ddelta, float* dA,
           float* dB, float* dC, float* dD, float* dz, float* ddelta_bias, int64_t Bsz, int64_t L, int64_t Dch,
           int64_t N, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_sizes(Bsz, L, Dch, N, dtype);
    if (rc != SS_OK) return rc;
    if ((D == nullptr) != (dD == nullptr) || (z == nullptr) != (dz == nullptr) ||
        (delta_bias == nullptr) != (ddelta_bias == nullptr))
        return SS_ERR_INVALID_PROBLEM;
    const bool empty = Bsz == 0 || L == 0 || Dch == 0;
    if (!empty && (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC))
        return SS_ERR_INVALID_PROBLEM;
    if (empty && Dch > 0 && N > 0 && !dA) return SS_ERR_INVALID_PROBLEM;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, dy, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                          workspace};
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
    if (ceil_div(Dch, 4) * Bsz * p.K >= (1ll << 31)) return SS_ERR_UNSUPPORTED;
    const BwdLayout w = bwd_layout2(p, Bsz, L, Dch, N);
    if (workspace_bytes < w.total || workspace == nullptr) return SS_ERR_WORKSPACE_TOO_SMALL;
    char* ws = static_cast<char*>(workspace);
    BwdArgs a;
    a.f.u = u; a.f.delta = delta; a.f.B = B; a.f.C = C; a.f.z = z;
    a.f.A = A; a.f.D = D; a.f.delta_bias = delta_bias;
    a.f.y = nullptr; a.f.last_state = nullptr;
    a.f.Bsz = Bsz; a.f.L = L; a.f.Dch = Dch; a.f.N = N;
    a.f.softplus = softplus ? 1 : 0;
    a.f.dtype = dtype;
    a.f.ws_fsum = reinterpret_cast<float*>(ws + w.fsum);
    a.dy = dy;
    a.du = du; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz;
    a.ddelta_bias = ddelta_bias;
    a.ws_rsum = reinterpret_cast<float*>(ws + w.rsum);
    a.ws_ckpt = reinterpret_cast<float*>(ws + w.ckpt);
    a.ws_bc = reinterpret_cast<float*>(ws + w.bc);
    a.ws_dA = reinterpret_cast<float*>(ws + w.dA);
    a.ws_dD = reinterpret_cast<float*>(ws + w.dD);
    a.ws_db = reinterpret_cast<float*>(ws + w.db);
    return launch_bwd2(a, p, st) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // extern "C"
