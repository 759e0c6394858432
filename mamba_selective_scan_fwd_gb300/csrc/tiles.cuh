// Tile staging helpers shared by the forward and backward scans: io
// elements held as 32-bit words (bf16 unpacks exactly to f32), vector loads
// of row runs of the [B, L, D] tensors, asynchronous copies into shared
// memory, and the f32 B / C staging rows whose state groups hold S values of
// B followed by S values of C.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "simd.cuh"

namespace ss {

// element j of a row held as 32-bit words (f32, bf16 or f16 io; both 16-bit
// types convert to f32 exactly)
template <typename T>
__device__ __forceinline__ float elem(const uint32_t* w, int j) {
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(w[j]);
    } else if constexpr (std::is_same<T, __half>::value) {
        const uint32_t v = w[j >> 1];
        return __half2float(__ushort_as_half((unsigned short)((j & 1) ? (v >> 16) : (v & 0xffffu))));
    } else {
        return (j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]);
    }
}

// Two f32 values rounded to nearest (ties to even) into one word of the
// 16-bit io type, lo | hi << 16.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (std::is_same<T, __half>::value) {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// Load NBYTES contiguous bytes (naturally aligned) into words.
template <int NBYTES, int NWORDS>
__device__ __forceinline__ void load_words(const void* p, uint32_t (&w)[NWORDS]) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int v = 0; v < NBYTES / 16; v++) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + v);
            w[4 * v] = q.x; w[4 * v + 1] = q.y; w[4 * v + 2] = q.z; w[4 * v + 3] = q.w;
        }
    } else if constexpr (NBYTES == 8) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = q.x; w[1] = q.y;
    } else if constexpr (NBYTES == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
    } else {
        w[0] = __ldg(reinterpret_cast<const unsigned short*>(p));
    }
}

// CNT consecutive elements of a [Bsz, L, Dch] io tensor at element offset
// off (channel c0): vector loads when the run is aligned and complete,
// element loads (zero-filled past Dch) otherwise.
template <typename T, int CNT, int RW>
__device__ __forceinline__ void load_run(const T* base, int64_t off, int64_t c0, int64_t Dch, bool fast,
                                         uint32_t (&w)[RW]) {
    if (fast) {
        load_words<CNT * (int)sizeof(T), RW>(base + off, w);
    } else {
#pragma unroll
        for (int i = 0; i < RW; i++) w[i] = 0u;
#pragma unroll
        for (int c = 0; c < CNT; c++) {
            if (c0 + c < Dch) {
                if constexpr (sizeof(T) == 4) {
                    w[c] = __ldg(reinterpret_cast<const unsigned int*>(base + off) + c);
                } else {
                    const uint32_t v = __ldg(reinterpret_cast<const unsigned short*>(base + off) + c);
                    w[c >> 1] |= (c & 1) ? (v << 16) : v;
                }
            }
        }
    }
}

// Load NBYTES (4, 8 or a multiple of 16) naturally aligned bytes of shared memory into words.
template <int NBYTES, int NWORDS>
__device__ __forceinline__ void lds_words(const void* p, uint32_t (&w)[NWORDS]) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int v = 0; v < NBYTES / 16; v++) {
            const uint4 q = reinterpret_cast<const uint4*>(p)[v];
            w[4 * v] = q.x; w[4 * v + 1] = q.y; w[4 * v + 2] = q.z; w[4 * v + 3] = q.w;
        }
    } else if constexpr (NBYTES == 8) {
        const uint2 q = *reinterpret_cast<const uint2*>(p);
        w[0] = q.x; w[1] = q.y;
    } else {
        w[0] = *reinterpret_cast<const unsigned int*>(p);
    }
}

// Store NWORDS words (NBYTES = 4, 8 or a multiple of 16 bytes) to naturally aligned shared memory.
template <int NBYTES, int NWORDS>
__device__ __forceinline__ void sts_words(void* p, const uint32_t* w) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int v = 0; v < NBYTES / 16; v++)
            reinterpret_cast<uint4*>(p)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    } else if constexpr (NBYTES == 8) {
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<unsigned int*>(p) = w[0];
    }
}

// S consecutive f32 values of shared memory (16-byte aligned when S = 4,
// 8-byte aligned when S = 2).
template <int S>
__device__ __forceinline__ void ld_f32(const float* p, float (&v)[S]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 f = *reinterpret_cast<const float4*>(p + q);
            v[q] = f.x; v[q + 1] = f.y; v[q + 2] = f.z; v[q + 3] = f.w;
        }
    } else if constexpr (S == 2) {
        const float2 f = *reinterpret_cast<const float2*>(p);
        v[0] = f.x; v[1] = f.y;
    } else {
        v[0] = p[0];
    }
}

// B and C values of one f32 state group (S floats of B, then S of C).
template <int S>
__device__ __forceinline__ void ld_bc_f32(const float* g, float (&Bv)[S], float (&Cv)[S]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int s = 0; s < S; s += 4) {
            const float4 b = *reinterpret_cast<const float4*>(g + s), c = *reinterpret_cast<const float4*>(g + S + s);
            Bv[s] = b.x; Bv[s + 1] = b.y; Bv[s + 2] = b.z; Bv[s + 3] = b.w;
            Cv[s] = c.x; Cv[s + 1] = c.y; Cv[s + 2] = c.z; Cv[s + 3] = c.w;
        }
    } else if constexpr (S == 2) {
        const float4 v = *reinterpret_cast<const float4*>(g);
        Bv[0] = v.x; Bv[1] = v.y; Cv[0] = v.z; Cv[1] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(g);
        Bv[0] = v.x; Cv[0] = v.y;
    }
}

// B values only of one f32 state group.
template <int S>
__device__ __forceinline__ void ld_b_f32(const float* g, float (&Bv)[S]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int s = 0; s < S; s += 4) {
            const float4 b = *reinterpret_cast<const float4*>(g + s);
            Bv[s] = b.x; Bv[s + 1] = b.y; Bv[s + 2] = b.z; Bv[s + 3] = b.w;
        }
    } else if constexpr (S == 2) {
        const float2 b = *reinterpret_cast<const float2*>(g);
        Bv[0] = b.x; Bv[1] = b.y;
    } else {
        Bv[0] = g[0];
    }
}

// Write a B or C row (N io values held as words) as f32 into the state groups
// of a step's staging row: group q holds floats q S .. q S + S of B, then of
// C.  A row past the chunk end is staged as zeros.
template <typename T, int N, int S, int NWd>
__device__ __forceinline__ void stage_bc_row_f32(float* row, int half, const uint32_t (&w)[NWd], bool valid) {
#pragma unroll
    for (int q = 0; q < N / S; q++) {
        float* dst = row + q * 2 * S + half * S;
        if constexpr (S % 4 == 0) {
#pragma unroll
            for (int s = 0; s < S; s += 4)
                *reinterpret_cast<float4*>(dst + s) =
                    valid ? make_float4(elem<T>(w, q * S + s), elem<T>(w, q * S + s + 1), elem<T>(w, q * S + s + 2),
                                        elem<T>(w, q * S + s + 3))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
#pragma unroll
            for (int s = 0; s < S; s++) dst[s] = valid ? elem<T>(w, q * S + s) : 0.f;
        }
    }
}

// Asynchronous global -> shared copy of NBYTES (4, 8 or a multiple of 16)
// bytes; both addresses are aligned to min(NBYTES, 16).  Completion is
// awaited per thread with cp_async_wait after cp_async_commit.
template <int NBYTES>
__device__ __forceinline__ void cp_async_bytes(void* dst, const void* src) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(dst);
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int q = 0; q < NBYTES; q += 16)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + q),
                         "l"(static_cast<const char*>(src) + q)
                         : "memory");
    } else {
        static_assert(NBYTES == 4 || NBYTES == 8, "cp.async copies 4, 8 or 16 bytes");
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(src), "n"(NBYTES) : "memory");
    }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

// Issue the copies of an f32 B or C row (N values at src) into the state
// groups of a step's staging row (the layout of stage_bc_row_f32), or zero
// the groups of a step past the chunk end.
template <typename T, int N, int S>
__device__ __forceinline__ void cp_async_bc_row(unsigned char* row, int half, const T* src, bool valid) {
    constexpr int GB = S * (int)sizeof(T);
    static_assert(GB >= 4, "a state group half of at least 4 bytes");
#pragma unroll
    for (int q = 0; q < N / S; q++) {
        unsigned char* dst = row + q * 2 * GB + half * GB;
        if (valid) {
            cp_async_bytes<GB>(dst, src + q * S);
        } else {
#pragma unroll
            for (int i = 0; i < GB; i += 4) *reinterpret_cast<unsigned int*>(dst + i) = 0u;
        }
    }
}

}  // namespace ss
