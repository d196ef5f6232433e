// dense_common.cuh -- pieces shared by the gated-delta-rule (dense) scan kernels:
// bf16 hi + lo splitting, bounded waits with a shared abort flag, and the
// blocked inverse A = (I + L)^-1 of a chunk's strictly lower 64 x 64 matrix L.
#pragma once

#include <cuda_bf16.h>

#include "sm100.cuh"

namespace hypic {
namespace dense {

using namespace sm100;

constexpr int kC = 64;    // tokens per chunk
constexpr int kLd = 68;   // padded row stride of the fp32 L / A work tiles (16-byte rows)

// x = hi + lo with both in bf16 (pairs packed for elements 2c, 2c+1)
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abortp) {
    if (*abortp) return false;
    if (!mbar_wait(bar, parity)) {
        *abortp = 1;
        return false;
    }
    return true;
}

__device__ __forceinline__ int exponent_of(float mx) {   // 2^e <= mx < 2^(e+1)
    if (!(mx > 0.f)) return 0;
    int ex;
    frexpf(mx, &ex);
    return ex - 1;
}

// Off-diagonal blocks of A at block distance DIST (16 x 16 blocks):
//   T = sum_{k=j}^{i-1} L_ik A_kj,  A_ij = -A_ii T,
// four adjacent columns of one row per task (16-byte loads of A and T).
// NT threads (pt = 0 .. NT-1) take part; named barrier BAR.
template <int DIST, int NT, int BAR, bool PACKED>
__device__ __forceinline__ void inverse_level(const float *Lw, float *Aw, float *Tw, int pt) {
    constexpr int NB = 4 - DIST;
    for (int task = pt; task < NB * 64; task += NT) {
        const int blk = task >> 6, r = (task >> 2) & 15, c4 = (task & 3) * 4;
        const int bi = blk + DIST, bj = bi - DIST;
        const float *lrow = Lw + (bi * 16 + r) * kLd + bj * 16;
        const float *acol = Aw + (bj * 16) * kLd + bj * 16 + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (PACKED) {
            // packed f32x2 FMAs (two columns an instruction), two partial sums per pair
            uint64_t a01[2] = {0, 0}, a23[2] = {0, 0};
#pragma unroll
            for (int k = 0; k < 16 * DIST; ++k) {
                const float lv = lrow[k];
                const uint64_t l2 = pk2(lv, lv);
                const float4 av = *reinterpret_cast<const float4 *>(acol + k * kLd);
                a01[k & 1] = fma2(l2, pk2(av.x, av.y), a01[k & 1]);
                a23[k & 1] = fma2(l2, pk2(av.z, av.w), a23[k & 1]);
            }
            upk2(add2(a01[0], a01[1]), acc.x, acc.y);
            upk2(add2(a23[0], a23[1]), acc.z, acc.w);
        } else {
#pragma unroll
            for (int k = 0; k < 16 * DIST; ++k) {
                const float lv = lrow[k];
                const float4 av = *reinterpret_cast<const float4 *>(acol + k * kLd);
                acc.x = fmaf(lv, av.x, acc.x);
                acc.y = fmaf(lv, av.y, acc.y);
                acc.z = fmaf(lv, av.z, acc.z);
                acc.w = fmaf(lv, av.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(Tw + blk * 256 + r * 16 + c4) = acc;
    }
    bar_sync(BAR, NT);
    for (int task = pt; task < NB * 64; task += NT) {
        const int blk = task >> 6, r = (task >> 2) & 15, c4 = (task & 3) * 4;
        const int bi = blk + DIST, bj = bi - DIST;
        const float *arow = Aw + (bi * 16 + r) * kLd + bi * 16;   // A_ii, zero above the diagonal
        const float *tcol = Tw + blk * 256 + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (PACKED) {
            uint64_t a01[2] = {0, 0}, a23[2] = {0, 0};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float av = arow[k];
                const uint64_t m2 = pk2(av, av);
                const float4 tv = *reinterpret_cast<const float4 *>(tcol + k * 16);
                a01[k & 1] = fma2(m2, pk2(tv.x, tv.y), a01[k & 1]);
                a23[k & 1] = fma2(m2, pk2(tv.z, tv.w), a23[k & 1]);
            }
            upk2(add2(a01[0], a01[1]), acc.x, acc.y);
            upk2(add2(a23[0], a23[1]), acc.z, acc.w);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float av = arow[k];
                const float4 tv = *reinterpret_cast<const float4 *>(tcol + k * 16);
                acc.x = fmaf(av, tv.x, acc.x);
                acc.y = fmaf(av, tv.y, acc.y);
                acc.z = fmaf(av, tv.z, acc.z);
                acc.w = fmaf(av, tv.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(Aw + (bi * 16 + r) * kLd + bj * 16 + c4) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    bar_sync(BAR, NT);
}

// A = (I + L)^-1 for the strictly lower 64 x 64 L in Lw (row stride kLd; entries
// on and above the diagonal are not read).  Diagonal 16 x 16 blocks by forward
// substitution in column (axpy) order -- one column per thread in registers, a
// dependent chain of 16 steps -- then three block levels.  ZERO_UPPER also
// writes the zero blocks above the diagonal (else the caller never reads them).
// Needs NT >= 128; Tw holds 3 x 256 floats.  Ends with a barrier.
// PACKED: the block levels with packed f32x2 FMAs (fewer instructions, more registers).
template <int NT, int BAR, bool ZERO_UPPER = true, bool PACKED = false>
__device__ __forceinline__ void tri_inverse(const float *Lw, float *Aw, float *Tw, int pt) {
    static_assert(NT >= 128, "one column per thread for the diagonal blocks, the rest zero the upper blocks");
    if (pt < 64) {
        const int b0 = (pt >> 4) * 16, jc = pt & 15, col = b0 + jc;
        float ac[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) ac[i] = i == jc ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
            // ac[k] is final here; push its contribution down the column
#pragma unroll
            for (int i = k + 1; i < 16; ++i) ac[i] = fmaf(-Lw[(b0 + i) * kLd + b0 + k], ac[k], ac[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Aw[(b0 + i) * kLd + col] = ac[i];
    } else if (ZERO_UPPER) {
        // zero the strictly upper off-diagonal blocks
        for (int e = pt - 64; e < 6 * 256; e += NT - 64) {
            const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            Aw[(bi * 16 + r) * kLd + bj * 16 + c] = 0.f;
        }
    }
    bar_sync(BAR, NT);
    inverse_level<1, NT, BAR, PACKED>(Lw, Aw, Tw, pt);
    inverse_level<2, NT, BAR, PACKED>(Lw, Aw, Tw, pt);
    inverse_level<3, NT, BAR, PACKED>(Lw, Aw, Tw, pt);
}

}  // namespace dense
}  // namespace hypic
