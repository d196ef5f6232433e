// scan_recurrent.cu -- token-by-token segment scan on CUDA cores, fp32.
//
// One CTA walks one (layer, segment, head) chain token by token, exactly the
// recurrence of the family (S_t = T_t S_{t-1} + beta_t k_t v_t^T, see hypic.h),
// keeping the state in registers.  It serves every family and the optional
// per-token output o_t = S_t^T q_t, and is the path for fp32 inputs, for
// scalar/diagonal scans that ask for o_t and for the KDA family.  The transition
// of the dense and KDA families is carried as exp(lambda) * M with M renormalised
// by exact powers of two (KDA's per-channel gates stay inside M).
//
// Thread layout: the state (and, for the dense and KDA families, M) is split by
// columns: thread (g, c) owns column c and rows [g*RPT, (g+1)*RPT).  A token
// is a rank-1 update of every column, so a thread needs only the scalar
// u_c = k^T X[:, c] (a reduction over its G row groups) and the broadcast key.
// M and S do not depend on each other, so for the families with M a chain takes
// two CTAs, one for the columns of M (and lambda) and one for those of S (and
// o_t): half the threads a CTA, two CTAs an SM whose per-token barriers do not
// wait for each other.
#include "internal.cuh"

namespace hypic {
namespace {

constexpr int kTB = 16;  // tokens staged in shared memory per round

// sum_r a[r] x[r] over RPT rows in four interleaved partial sums (a fixed order:
// four independent FMA chains instead of one of RPT)
template <int RPT>
__device__ __forceinline__ float dot_rows(const float *a, const float (&x)[RPT]) {
    static_assert(RPT % 4 == 0, "rows in fours");
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
    for (int r = 0; r < RPT; r += 4) {
        p0 = fmaf(a[r], x[r], p0);
        p1 = fmaf(a[r + 1], x[r + 1], p1);
        p2 = fmaf(a[r + 2], x[r + 2], p2);
        p3 = fmaf(a[r + 3], x[r + 3], p3);
    }
    return (p0 + p1) + (p2 + p3);
}

__device__ __forceinline__ void kahan_add(float &sum, float &comp, float v) {
    const float y = v - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

// LIST: the units are a.unit_list[0 .. *a.unit_count), walked in a grid-stride loop
template <int FAM, int DK, typename TIn, bool LIST = false>
__global__ void __launch_bounds__(256, 2) scan_recurrent_kernel(const ScanArgs a) {
    constexpr int RPT = DK == 128 ? 64 : 32;   // rows per thread
    constexpr int G = DK / RPT;              // row groups
    constexpr bool kDense = FAM == HYPIC_DENSE || FAM == HYPIC_KDA;   // erasing update, M columns
    constexpr bool kKda = FAM == HYPIC_KDA;
    constexpr bool kDiag = FAM == HYPIC_DIAG || FAM == HYPIC_KDA;     // a gate per channel
    const int DV = a.dv;
    const bool mpart = kDense && (blockIdx.x & 1) == 0;  // this CTA: the columns of M (else of S)
    const int NCOL = mpart ? DK : DV;
    const int NT = NCOL * G;                             // working threads
    const int NTB = (int)blockDim.x;                     // all threads (max(DK, DV) * G with M)
    const int tid = threadIdx.x;
    const bool active = tid < NT;
    const int c = tid % NCOL, g = tid / NCOL;
    const int row0 = active ? g * RPT : 0;
    const bool mcol = mpart;                             // column of M
    const int scol = c;                                  // column of S (if !mcol)
    const bool want_o = a.o_out != nullptr;
    const bool o_here = want_o && !mpart;                // this CTA writes o_t

    extern __shared__ float smem[];
    float *sk = smem;                                    // [kTB][DK]
    float *sv = sk + kTB * DK;                           // [kTB][DV]
    float *sq = sv + kTB * DV;                           // [kTB][DK] if want_o
    float *sa = sq + (want_o ? kTB * DK : 0);            // [kTB][DK] diag, else [kTB]
    float *sb = sa + kTB * (kDiag ? DK : 1);             // [kTB]
    float *red = sb + kTB;                               // [2][G][NCOL]
    float *redo = red + 2 * G * NCOL;                    // [G][DV]
    float *redm = redo + G * DV;                         // [32]

    // one unit per CTA (pair of CTAs with M), or with a unit list the listed units in a
    // grid-stride loop
    const int first = kDense ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int stride = kDense ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int n_list = LIST ? *a.unit_count : 0;
    for (int it = first; !LIST || it < n_list; it += stride) {
    const int unit = LIST ? a.unit_list[it] : it;
    const int h = unit % a.H;
    const int seg = (unit / a.H) % a.n_seg;
    const int l = unit / (a.H * a.n_seg);

    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    if (!(t0 >= 0 && t0 <= t1 && t1 <= a.N)) {
        if (tid == 0) flag_index_error(a.d_err);
        t0 = t1 = 0;
    }

    float x[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) x[r] = (mcol && active && row0 + r == c) ? 1.f : 0.f;
    float lam_sum = 0.f, lam_comp = 0.f;
    int lam_exp = 0;   // power-of-two exponent moved out of M

    const TIn *Kp = static_cast<const TIn *>(a.k);
    const TIn *Vp = static_cast<const TIn *>(a.v);
    const TIn *Qp = static_cast<const TIn *>(a.q);
    TIn *Op = static_cast<TIn *>(a.o_out);
    const int64_t layer_row0 = (int64_t)l * a.N;

    for (int64_t tb = t0; tb < t1; tb += kTB) {
        const int nt = (int)((t1 - tb) < kTB ? (t1 - tb) : kTB);
        __syncthreads();
        for (int i = tid; i < nt * DK; i += NTB) {
            const int tt = i / DK, d = i % DK;
            const int64_t row = (layer_row0 + tb + tt) * a.H + h;
            sk[tt * DK + d] = to_f32(Kp[row * DK + d]);
            if (o_here) sq[tt * DK + d] = to_f32(Qp[row * DK + d]);
            if (kDiag) sa[tt * DK + d] = a.alpha[row * DK + d];
        }
        if (!mpart)
            for (int i = tid; i < nt * DV; i += NTB) {
                const int tt = i / DV, d = i % DV;
                const int64_t row = (layer_row0 + tb + tt) * a.H + h;
                sv[tt * DV + d] = to_f32(Vp[row * DV + d]);
            }
        for (int i = tid; i < nt; i += NTB) {
            const int64_t row = (layer_row0 + tb + i) * a.H + h;
            if (!kDiag) sa[i] = a.alpha[row];
            sb[i] = a.beta ? a.beta[row] : 1.f;
        }
        __syncthreads();

        for (int tt = 0; tt < nt; ++tt) {
            const float *kt = sk + tt * DK + row0;
            const float b = sb[tt];
            if (kKda) {
                // T_t = diag(alpha) (I - beta k k^T): erase, then gate each row
                const float *at = sa + tt * DK + row0;
                const float p = dot_rows<RPT>(kt, x);
                float u = p;
                if (G > 1) {
                    float *rb = red + (tt & 1) * G * NCOL;
                    if (active) rb[g * NCOL + c] = p;
                    __syncthreads();
                    u = 0.f;
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) u += rb[gg * NCOL + c];
                }
                const float w = -b * u;
                if (mcol) {
#pragma unroll
                    for (int r = 0; r < RPT; ++r) x[r] = at[r] * fmaf(kt[r], w, x[r]);
                } else {
                    const float bv = b * sv[tt * DV + scol];
#pragma unroll
                    for (int r = 0; r < RPT; ++r) x[r] = fmaf(kt[r], bv, at[r] * fmaf(kt[r], w, x[r]));
                }
            } else if (kDense) {
                const float al = sa[tt];
                const float p = dot_rows<RPT>(kt, x);
                float u = p;
                if (G > 1) {
                    float *rb = red + (tt & 1) * G * NCOL;
                    if (active) rb[g * NCOL + c] = p;
                    __syncthreads();
                    u = 0.f;
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) u += rb[gg * NCOL + c];
                }
                if (mcol) {
                    // M <- M - beta k (k^T M)
                    const float w = -b * u;
#pragma unroll
                    for (int r = 0; r < RPT; ++r) x[r] = fmaf(kt[r], w, x[r]);
                } else {
                    // S <- alpha (S - beta k (k^T S)) + beta k v^T = alpha S + k (beta (v - alpha u))^T
                    const float w = b * (sv[tt * DV + scol] - al * u);
#pragma unroll
                    for (int r = 0; r < RPT; ++r) x[r] = fmaf(kt[r], w, al * x[r]);
                }
                if (tid == 0) kahan_add(lam_sum, lam_comp, logf(al));
            } else if (!kDiag) {
                const float al = sa[tt];
                const float w = b * sv[tt * DV + scol];
#pragma unroll
                for (int r = 0; r < RPT; ++r) x[r] = fmaf(kt[r], w, al * x[r]);
                if (tid == 0) kahan_add(lam_sum, lam_comp, logf(al));
            } else {
                const float *at = sa + tt * DK;
                const float w = b * sv[tt * DV + scol];
#pragma unroll
                for (int r = 0; r < RPT; ++r) x[r] = fmaf(kt[r], w, at[row0 + r] * x[r]);
                if (tid < DK) kahan_add(lam_sum, lam_comp, logf(at[tid]));
            }
            if (o_here) {
                float po = 0.f;
                if (!mcol) po = dot_rows<RPT>(sq + tt * DK + row0, x);
                const int64_t orow = (layer_row0 + tb + tt) * a.H + h;
                if (G > 1) {
                    __syncthreads();
                    if (active) redo[g * DV + scol] = po;
                    __syncthreads();
                    if (!mcol && g == 0) {
                        float s = 0.f;
#pragma unroll
                        for (int gg = 0; gg < G; ++gg) s += redo[gg * DV + scol];
                        Op[orow * DV + scol] = from_f32<TIn>(s);
                    }
                } else if (active) {
                    Op[orow * DV + scol] = from_f32<TIn>(po);
                }
            }
        }

        if (kDense && mpart) {
            // keep max|M| in [1, 2) with exact power-of-two scaling
            float mx = 0.f;
            if (active) {
#pragma unroll
                for (int r = 0; r < RPT; ++r) mx = fmaxf(mx, fabsf(x[r]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            __syncthreads();
            if ((tid & 31) == 0) redm[tid >> 5] = mx;
            __syncthreads();
            mx = 0.f;
            for (int w = 0; w < NTB / 32; ++w) mx = fmaxf(mx, redm[w]);
            if (mx > 0.f && (mx < 1.f || mx >= 2.f)) {
                int ex;
                frexpf(mx, &ex);
                const int e = ex - 1;
                const float sc = ldexpf(1.f, -e);
                if (mcol) {
#pragma unroll
                    for (int r = 0; r < RPT; ++r) x[r] *= sc;
                }
                lam_exp += e;
            }
        }
    }

    const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
    if (!active) {
    } else if (!mcol) {
        float *So = a.S_out + u_out * DK * DV;
#pragma unroll
        for (int r = 0; r < RPT; ++r) So[(int64_t)(row0 + r) * DV + scol] = x[r];
    } else {
        float *Mo = a.M_out + u_out * DK * DK;
#pragma unroll
        for (int r = 0; r < RPT; ++r) Mo[(int64_t)(row0 + r) * DK + c] = x[r];
    }
    if (FAM == HYPIC_DIAG) {   // lambda per channel
        if (tid < DK) a.lam_out[u_out * DK + tid] = lam_sum;
    } else if (tid == 0 && (!kDense || mpart)) {   // with M: the M CTA, which holds the exponent
        const double lam = (double)lam_sum + (double)lam_exp * 0.69314718055994530942;
        a.lam_out[u_out] = (float)lam;
    }
    if (!LIST) break;
    __syncthreads();   // the next listed unit reuses the shared tiles
    }
}

template <int FAM, int DK, typename TIn>
cudaError_t launch_one(const ScanArgs &a, cudaStream_t s) {
    constexpr int RPT = DK == 128 ? 64 : 32;
    constexpr int G = DK / RPT;
    constexpr bool kM = FAM == HYPIC_DENSE || FAM == HYPIC_KDA;
    const int ncol = kM ? (DK > a.dv ? DK : a.dv) : a.dv;   // columns of the wider CTA
    const int nt = ncol * G;
    const bool want_o = a.o_out != nullptr;
    size_t floats = (size_t)kTB * DK + (size_t)kTB * a.dv + (want_o ? (size_t)kTB * DK : 0) +
                    (size_t)kTB * (FAM == HYPIC_DIAG || FAM == HYPIC_KDA ? DK : 1) + kTB + 2 * G * ncol + G * a.dv + 32;
    const size_t smem = floats * sizeof(float);
    auto kern = scan_recurrent_kernel<FAM, DK, TIn>;
    // listed units: only the KDA scan's steep chunks (d = 128, bf16) use them
    if (a.unit_list) {
        if constexpr (FAM == HYPIC_KDA && DK == 128 && sizeof(TIn) == 2) kern = scan_recurrent_kernel<FAM, DK, TIn, true>;
        else return cudaErrorInvalidValue;
    }
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    if (a.unit_list) {   // a few listed units at most: two CTAs (pairs with M) per SM walk them
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 148;
        units = units < 2 * sms ? units : 2 * sms;
    }
    kern<<<(unsigned)(units * (kM ? 2 : 1)), nt, smem, s>>>(a);
    return cudaGetLastError();
}

template <int FAM, typename TIn>
cudaError_t launch_dk(const ScanArgs &a, cudaStream_t s) {
    switch (a.dk) {
        case 32: return launch_one<FAM, 32, TIn>(a, s);
        case 64: return launch_one<FAM, 64, TIn>(a, s);
        case 128: return launch_one<FAM, 128, TIn>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t launch_fam(const ScanArgs &a, cudaStream_t s) {
    switch (a.fam) {
        case HYPIC_SCALAR: return launch_dk<HYPIC_SCALAR, TIn>(a, s);
        case HYPIC_DIAG: return launch_dk<HYPIC_DIAG, TIn>(a, s);
        case HYPIC_DENSE: return launch_dk<HYPIC_DENSE, TIn>(a, s);
        case HYPIC_KDA: return launch_dk<HYPIC_KDA, TIn>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_recurrent(const ScanArgs &a, cudaStream_t s) {
    if ((int64_t)a.n_layers * a.n_seg * a.H == 0) return cudaSuccess;
    return a.in_dtype == HYPIC_BF16 ? launch_fam<__nv_bfloat16>(a, s) : launch_fam<float>(a, s);
}

}  // namespace hypic
