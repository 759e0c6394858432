// Tile staging helpers shared by the forward and backward scans: io
// elements held as 32-bit words (bf16 unpacks exactly to f32), vector loads
// of row runs of the [B, L, D] tensors, and the raw B / C staging rows whose
// state groups hold S values of B followed by S values of C.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "simd.cuh"

namespace ss {

// element j of a row held as 32-bit words
template <typename T>
__device__ __forceinline__ float elem(const uint32_t* w, int j) {
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(w[j]);
    } else {
        return (j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]);
    }
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

// B and C values of one state group (S raw io values of B, then S of C) as floats.
template <typename T, int S>
__device__ __forceinline__ void ld_bc(const unsigned char* g, float (&Bv)[S], float (&Cv)[S]) {
    constexpr int NB = 2 * S * (int)sizeof(T), NW = NB / 4;
    uint32_t w[NW];
    lds_words<NB, NW>(g, w);
#pragma unroll
    for (int s = 0; s < S; s++) {
        Bv[s] = elem<T>(w, s);
        Cv[s] = elem<T>(w, S + s);
    }
}

// Copy a B or C row (N io values held as words) into the state groups of a
// step's staging row: group q gets values q S .. q S + S at byte offset
// q * 2 S esz + half * S esz (half 0: B, 1: C).  A row past the chunk end is
// staged as zeros.
template <typename T, int N, int S, int NWd>
__device__ __forceinline__ void stage_bc_row(unsigned char* row, int half, const uint32_t (&w)[NWd], bool valid) {
    constexpr int ESZ = (int)sizeof(T);
    constexpr int GB = S * ESZ;  // bytes of one half of a group
    if constexpr (GB % 4 == 0) {
        constexpr int GW = GB / 4;
#pragma unroll
        for (int q = 0; q < N / S; q++) {
            uint32_t v[GW];
#pragma unroll
            for (int i = 0; i < GW; i++) v[i] = valid ? w[q * GW + i] : 0u;
            sts_words<GB, GW>(row + q * 2 * GB + half * GB, v);
        }
    } else {
        // S = 1 with 2-byte values: one element per group half
#pragma unroll
        for (int q = 0; q < N; q++) {
            const uint32_t word = w[q >> 1];
            const unsigned short v = (unsigned short)((q & 1) ? (word >> 16) : (word & 0xffffu));
            *reinterpret_cast<unsigned short*>(row + q * 2 * GB + half * GB) = valid ? v : (unsigned short)0;
        }
    }
}

// B values only of one state group (the first half of the group).
template <typename T, int S>
__device__ __forceinline__ void ld_b(const unsigned char* g, float (&Bv)[S]) {
    constexpr int NB = S * (int)sizeof(T), NW = NB >= 4 ? NB / 4 : 1;
    if constexpr (NB >= 4) {
        uint32_t w[NW];
        lds_words<NB, NW>(g, w);
#pragma unroll
        for (int s = 0; s < S; s++) Bv[s] = elem<T>(w, s);
    } else {
        Bv[0] = bf16lo(*reinterpret_cast<const unsigned short*>(g));
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

// Issue the copies of a B or C row (N io values at src) into the state
// groups of a step's staging row (the layout of stage_bc_row), or zero the
// groups of a step past the chunk end.  Needs S * esz >= 4 bytes.
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
