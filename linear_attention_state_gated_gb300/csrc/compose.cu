// compose.cu -- S = T_C S_prev + S_C (single step, batched) and the chained
// combine S <- T_p S + S_p over pool entries, for all three families.
//
// Scalar / diagonal: T is a row scaling exp(lambda_row), so every row of S
// composes independently -- pure streaming with 16-byte loads and stores.
// Dense: T = exp(lambda) M is a dk x dk matrix and each step is a small fp32
// GEMM per head, register-tiled on CUDA cores; one CTA owns one head so that
// S_out may alias S_prev.
#include "internal.cuh"

namespace hypic {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float4 axpy4(float s, float4 x, float4 y) {
    return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}

// ---------------------------------------------------------------- scalar/diag

// One CTA per (item, head): S_out = exp(lam) S_prev + S_C, row-wise scale.
template <bool kDiag>
__global__ void __launch_bounds__(256) compose_sd_kernel(const ComposeArgs a) {
    __shared__ float row_scale[128];
    const int DK = a.dk, DV = a.dv;
    const int64_t u = blockIdx.x;
    const int row4_shift = DV == 128 ? 5 : (DV == 64 ? 4 : 3);
    const int per4 = (DK * DV) >> 2;
    if (threadIdx.x < DK) {
        const float lam = kDiag ? a.lam[u * DK + threadIdx.x] : a.lam[u];
        row_scale[threadIdx.x] = expf(lam);
        if (a.lam_out) {
            if (kDiag)
                a.lam_out[u * DK + threadIdx.x] = lam + a.lam_prev[u * DK + threadIdx.x];
            else if (threadIdx.x == 0)
                a.lam_out[u] = lam + a.lam_prev[u];
        }
    }
    __syncthreads();
    const float4 *C = reinterpret_cast<const float4 *>(a.S_C) + u * per4;
    const float4 *P = a.S_prev ? reinterpret_cast<const float4 *>(a.S_prev) + u * per4 : nullptr;
    float4 *O = reinterpret_cast<float4 *>(a.S_out) + u * per4;
    constexpr int U = 4;
    for (int base = threadIdx.x; base < per4; base += U * 256) {
        float4 c[U], p[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int j = base + i * 256;
            if (j < per4) {
                c[i] = C[j];
                p[i] = P ? P[j] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int j = base + i * 256;
            if (j < per4) O[j] = axpy4(row_scale[j >> row4_shift], p[i], c[i]);
        }
    }
}

// ---------------------------------------------------------------- dense GEMM

// out[DM x DN] = scale * (A[DM x DM] B[DM x DN]) (+ C), one CTA per head,
// 256 threads as 16 x 16; thread (ty, tx) owns rows ty*TM + i and columns
// tx + 16 j.  A is staged transposed in chunks of KC columns.
template <int DM, int DN>
struct HeadGemm {
    static constexpr int TM = DM / 16, TN = DN / 16, KC = 32;
    static constexpr int AS_LD = DM + 4;   // padded; keeps float4 rows aligned

    // acc += A[:, k0:k0+KC] * B[k0:k0+KC, :], B read from `Bsrc` with leading dim DN
    // (global or shared), A staged through `As`.
    template <bool kBShared>
    static __device__ __forceinline__ void run(const float *A, const float *Bsrc, float *As,
                                               float (&acc)[TM][TN]) {
        const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
        for (int k0 = 0; k0 < DM; k0 += KC) {
            __syncthreads();
            // stage A[m][k0 + kk] -> As[kk][m]
            for (int i = tid; i < DM * KC; i += 256) {
                const int kk = i & (KC - 1), m = i / KC;
                As[kk * AS_LD + m] = A[(int64_t)m * DM + k0 + kk];
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < KC; ++kk) {
                float af[TM], bf[TN];
                if constexpr (TM % 4 == 0) {
#pragma unroll
                    for (int i = 0; i < TM; i += 4) {
                        const float4 t = *reinterpret_cast<const float4 *>(&As[kk * AS_LD + ty * TM + i]);
                        af[i] = t.x; af[i + 1] = t.y; af[i + 2] = t.z; af[i + 3] = t.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < TM; ++i) af[i] = As[kk * AS_LD + ty * TM + i];
                }
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const float *bp = Bsrc + (int64_t)(k0 + kk) * DN + tx + 16 * j;
                    bf[j] = kBShared ? *bp : __ldg(bp);
                }
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
            }
        }
    }
};

// Dense single-step compose.  Part 0: S_out = exp(lam) M S_prev + S_C.
// Part 1 (operator requested): M_out = M M_prev renormalised, lam_out.
// Part = blockIdx.y + y0.
template <int D, int DV>
__global__ void __launch_bounds__(256) compose_dense_kernel(const ComposeArgs a, const int y0) {
    extern __shared__ __align__(16) float smem[];
    float *As = smem;
    __shared__ float redm[8];
    const int64_t u = blockIdx.x;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const float *M = a.M + u * D * D;
    if (blockIdx.y + y0 == 0) {
        using Gm = HeadGemm<D, DV>;
        float acc[Gm::TM][Gm::TN] = {};
        Gm::template run<false>(M, a.S_prev + u * D * DV, As, acc);
        __syncthreads();   // every read of S_prev of this head is done before any write
        const float sc = expf(a.lam[u]);
        const float *C = a.S_C + u * D * DV;
        float *O = a.S_out + u * D * DV;
#pragma unroll
        for (int i = 0; i < Gm::TM; ++i)
#pragma unroll
            for (int j = 0; j < Gm::TN; ++j) {
                const int64_t idx = (int64_t)(ty * Gm::TM + i) * DV + tx + 16 * j;
                O[idx] = fmaf(sc, acc[i][j], C[idx]);
            }
    } else {
        using Gm = HeadGemm<D, D>;
        float acc[Gm::TM][Gm::TN] = {};
        Gm::template run<false>(M, a.M_prev + u * D * D, As, acc);
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < Gm::TM; ++i)
#pragma unroll
            for (int j = 0; j < Gm::TN; ++j) mx = fmaxf(mx, fabsf(acc[i][j]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if ((tid & 31) == 0) redm[tid >> 5] = mx;
        __syncthreads();
        mx = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) mx = fmaxf(mx, redm[w]);
        int e = 0;
        if (mx > 0.f) {
            int ex;
            frexpf(mx, &ex);
            e = ex - 1;
        }
        const float sc = ldexpf(1.f, -e);
        float *O = a.M_out + u * D * D;
#pragma unroll
        for (int i = 0; i < Gm::TM; ++i)
#pragma unroll
            for (int j = 0; j < Gm::TN; ++j)
                O[(int64_t)(ty * Gm::TM + i) * D + tx + 16 * j] = acc[i][j] * sc;
        if (tid == 0) {
            const double lam = (double)a.lam[u] + (double)a.lam_prev[u] + (double)e * (double)kLn2;
            a.lam_out[u] = (float)lam;
        }
    }
}

// ---------------------------------------------------------------- chains

__device__ __forceinline__ int clamp_len(const ChainArgs &a, int r) {
    int n = a.chain_len[r];
    if (n < 0 || n > a.max_chain) {
        flag_index_error(a.d_err);
        n = n < 0 ? 0 : a.max_chain;
    }
    return n;
}

__device__ __forceinline__ int clamp_idx(const ChainArgs &a, int r, int j) {
    int p = a.seg_idx ? a.seg_idx[(int64_t)r * a.max_chain + j] : a.seg_first[r] + j;
    if (p < 0 || p >= a.P) {
        flag_index_error(a.d_err);
        p = p < 0 ? 0 : a.P - 1;
    }
    return p;
}

// One CTA per (request, layer, head); the state lives in registers, 16-byte
// vectors, and each pool entry is read exactly once.
template <bool kDiag>
__global__ void __launch_bounds__(256) chain_sd_kernel(const ChainArgs a) {
    constexpr int MAXV = 16;   // float4 per thread for a 128 x 128 state
    const int DK = a.dk, DV = a.dv;
    const int per4 = (DK * DV) >> 2;
    const int row4_shift = DV == 128 ? 5 : (DV == 64 ? 4 : 3);
    const int64_t u = blockIdx.x;                  // (r * Lyr + l) * H + h
    const int r = (int)(u / ((int64_t)a.n_layers * a.H));
    const int64_t lh = u % ((int64_t)a.n_layers * a.H);
    const int tid = threadIdx.x;
    float4 s[MAXV];
    const float4 *init = a.S_init ? reinterpret_cast<const float4 *>(a.S_init) + u * per4 : nullptr;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int j = tid + i * 256;
        s[i] = (init && j < per4) ? init[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __shared__ float row_scale[2][128];   // exp(lambda_row) of the current step, double-buffered
    const int n = clamp_len(a, r);
    for (int c = 0; c < n; ++c) {
        const int p = clamp_idx(a, r, c);
        const int64_t e = (int64_t)p * a.n_layers * a.H + lh;   // pool entry of this layer/head
        const float4 *Sp = reinterpret_cast<const float4 *>(a.pool_S) + e * per4;
        float4 x[MAXV];
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int j = tid + i * 256;
            if (j < per4) x[i] = __ldcs(Sp + j);
        }
        if (!kDiag) {
            const float sc = expf(a.pool_lam[e]);
#pragma unroll
            for (int i = 0; i < MAXV; ++i)
                if (tid + i * 256 < per4) s[i] = axpy4(sc, s[i], x[i]);
        } else if (DV == 128) {
            // float4 slot i of warp w covers row w + 8 i: 16 lanes compute the 16
            // row scales of the warp, shuffles hand them out (no block barrier)
            const int w = tid >> 5, lane = tid & 31;
            const int row = w + 8 * lane;
            const float ex = (lane < 16 && row < DK) ? expf(a.pool_lam[e * DK + row]) : 0.f;
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                const float sc = __shfl_sync(0xffffffffu, ex, i);
                if (tid + i * 256 < per4) s[i] = axpy4(sc, s[i], x[i]);
            }
        } else {
            float *rs = row_scale[c & 1];
            if (tid < DK) rs[tid] = expf(a.pool_lam[e * DK + tid]);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                const int j = tid + i * 256;
                if (j < per4) s[i] = axpy4(rs[j >> row4_shift], s[i], x[i]);
            }
        }
    }
    float4 *O = reinterpret_cast<float4 *>(a.S_out) + u * per4;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int j = tid + i * 256;
        if (j < per4) O[j] = s[i];
    }
}

// Dense chain: one CTA per (request, layer, head), S kept in shared memory,
// each step S <- exp(lam_p) M_p S + S_p as a register-tiled fp32 GEMM.  Operator
// mode (a.op, DV = D): S <- M_p S from I, brought back to max in [1, 2) by a power
// of two every 4 steps; the exponent goes to lam_out.
template <int D, int DV>
__global__ void __launch_bounds__(256) chain_dense_kernel(const ChainArgs a) {
    using Gm = HeadGemm<D, DV>;
    extern __shared__ __align__(16) float smem[];
    float *Ss = smem;                       // [D][DV]
    float *As = smem + D * DV;              // [KC][D + 4]
    const int64_t u = blockIdx.x;
    const int r = (int)(u / ((int64_t)a.n_layers * a.H));
    const int64_t lh = u % ((int64_t)a.n_layers * a.H);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    for (int i = tid; i < D * DV; i += 256)
        Ss[i] = a.op ? (i / DV == i % DV ? 1.f : 0.f) : (a.S_init ? a.S_init[u * D * DV + i] : 0.f);
    __shared__ float wmax[8];
    int op_exp = 0;
    const int n = clamp_len(a, r);
    for (int c = 0; c < n; ++c) {
        const int p = clamp_idx(a, r, c);
        const int64_t e = (int64_t)p * a.n_layers * a.H + lh;
        float acc[Gm::TM][Gm::TN] = {};
        Gm::template run<true>(a.pool_M + e * D * D, Ss, As, acc);
        const float sc = a.op ? 1.f : expf(a.pool_lam[e]);
        const float *Sp = a.pool_S + e * D * DV;
        __syncthreads();   // all reads of the old state are done
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < Gm::TM; ++i)
#pragma unroll
            for (int j = 0; j < Gm::TN; ++j) {
                const int idx = (ty * Gm::TM + i) * DV + tx + 16 * j;
                Ss[idx] = a.op ? acc[i][j] : fmaf(sc, acc[i][j], __ldcs(Sp + idx));
                mx = fmaxf(mx, fabsf(acc[i][j]));
            }
        if (a.op && (c & 3) == 3 && c + 1 < n) {   // one power of two for the whole matrix
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if ((tid & 31) == 0) wmax[tid >> 5] = mx;
            __syncthreads();
            mx = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wmax[w]);
            if (mx > 0.f && (mx < 1.f || mx >= 2.f)) {
                int ex;
                frexpf(mx, &ex);
                const float scl = ldexpf(1.f, 1 - ex);
#pragma unroll
                for (int i = 0; i < Gm::TM; ++i)
#pragma unroll
                    for (int j = 0; j < Gm::TN; ++j) Ss[(ty * Gm::TM + i) * DV + tx + 16 * j] *= scl;
                op_exp += ex - 1;
            }
            __syncthreads();   // the scaled state is in, wmax is read
        }
    }
    __syncthreads();
    for (int i = tid; i < D * DV; i += 256) a.S_out[u * D * DV + i] = Ss[i];
    if (a.op && tid == 0) a.lam_out[u] = (float)op_exp;
}

template <int D, int DV>
cudaError_t launch_dense_compose(const ComposeArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)HeadGemm<D, D>::KC * (D + 4) * sizeof(float);
    const int y0 = a.S_prev ? 0 : 1;
    const int parts = (a.S_prev ? 1 : 0) + (a.lam_out ? 1 : 0);
    if (parts == 0) return cudaSuccess;
    dim3 grid((unsigned)((int64_t)a.n * a.H), parts);
    compose_dense_kernel<D, DV><<<grid, 256, smem, s>>>(a, y0);
    return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_dense_chain(const ChainArgs &a, cudaStream_t s) {
    const size_t smem = ((size_t)D * DV + (size_t)HeadGemm<D, DV>::KC * (D + 4)) * sizeof(float);
    auto kern = chain_dense_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((int64_t)a.R * a.n_layers * a.H), 256, smem, s>>>(a);
    return cudaGetLastError();
}

template <template <int, int> class F, typename Args>
cudaError_t dispatch_dd(const Args &a, cudaStream_t s, int dk, int dv) {
#define HYPIC_DD(K, V) if (dk == K && dv == V) return F<K, V>::go(a, s);
    HYPIC_DD(32, 32) HYPIC_DD(32, 64) HYPIC_DD(32, 128)
    HYPIC_DD(64, 32) HYPIC_DD(64, 64) HYPIC_DD(64, 128)
    HYPIC_DD(128, 32) HYPIC_DD(128, 64) HYPIC_DD(128, 128)
#undef HYPIC_DD
    return cudaErrorInvalidValue;
}

template <int D, int DV> struct DenseComposeF {
    static cudaError_t go(const ComposeArgs &a, cudaStream_t s) { return launch_dense_compose<D, DV>(a, s); }
};
template <int D, int DV> struct DenseChainF {
    static cudaError_t go(const ChainArgs &a, cudaStream_t s) { return launch_dense_chain<D, DV>(a, s); }
};

}  // namespace

cudaError_t launch_compose(const ComposeArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.n * a.H;
    if (units == 0) return cudaSuccess;
    if (a.fam == HYPIC_DENSE) {
        if (a.S_prev && a.dk == 128 && a.dv == 128) {
            // the state on the tensor cores: a one-step chain per item, pool entry = item
            ChainArgs c{};
            c.fam = HYPIC_DENSE;
            c.R = a.n;
            c.n_layers = 1;
            c.H = a.H;
            c.dk = c.dv = 128;
            c.max_chain = 1;
            c.P = a.n;
            c.pool_lam = a.lam;
            c.pool_M = a.M;
            c.pool_S = a.S_C;
            c.S_init = a.S_prev;
            c.S_out = a.S_out;
            if (chain_dense_tc_supported(c)) {
                cudaError_t e = launch_chain_dense_tc(c, s);
                if (e != cudaSuccess || !a.lam_out) return e;
                ComposeArgs b = a;   // then the operator T(C1.C2) alone
                b.S_prev = nullptr;
                return dispatch_dd<DenseComposeF>(b, s, a.dk, a.dv);
            }
        }
        if (!a.S_prev) {
            // no previous state: S_out = S_C (a copy); only the operator needs the GEMM
            ComposeArgs b = a;
            b.lam_out = nullptr;
            compose_sd_kernel<false><<<(unsigned)units, 256, 0, s>>>(b);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        return dispatch_dd<DenseComposeF>(a, s, a.dk, a.dv);
    }
    if (a.fam == HYPIC_DIAG)
        compose_sd_kernel<true><<<(unsigned)units, 256, 0, s>>>(a);
    else
        compose_sd_kernel<false><<<(unsigned)units, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// Composed prefix, last pass: lambda of the group = sum of its entries' lambdas
// (double); for dense / kda also the exponent the operator chain took out and the
// final power of two that brings max|M| into [1, 2).  One CTA per (request, layer, head).
template <bool kM, bool kDiag>
__global__ void __launch_bounds__(256) prefix_finish_kernel(const ChainArgs a, float *lam_out, float *M_out) {
    const int64_t u = blockIdx.x;
    const int r = (int)(u / ((int64_t)a.n_layers * a.H));
    const int64_t lh = u % ((int64_t)a.n_layers * a.H);
    const int tid = threadIdx.x;
    const int nl = kDiag ? a.dk : 1;
    const int n = clamp_len(a, r);
    __shared__ double lsum[128];
    __shared__ float wmax[8];
    for (int x = tid; x < nl; x += 256) {
        double sum = 0.0;
        for (int c = 0; c < n; ++c) {
            const int64_t e = (int64_t)clamp_idx(a, r, c) * a.n_layers * a.H + lh;
            sum += (double)a.pool_lam[e * nl + x];
        }
        if (kM) lsum[x] = sum;
        else lam_out[u * nl + x] = (float)sum;
    }
    if (!kM) return;
    const int64_t DD = (int64_t)a.dk * a.dk;
    float *M = M_out + u * DD;
    const float E = lam_out[u];   // the operator chain's exponent
    float mx = 0.f;
    for (int64_t i = tid; i < DD; i += 256) mx = fmaxf(mx, fabsf(M[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((tid & 31) == 0) wmax[tid >> 5] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wmax[w]);
    int f = 0;
    if (mx > 0.f) {
        int ex;
        frexpf(mx, &ex);
        f = ex - 1;
    }
    const float scl = ldexpf(1.f, -f);
    for (int64_t i = tid; i < DD; i += 256) M[i] *= scl;
    if (tid == 0) lam_out[u] = (float)(lsum[0] + ((double)E + (double)f) * (double)kLn2);
}

cudaError_t launch_compose_prefix(const ChainArgs &a0, float *lam_out, float *M_out, cudaStream_t s) {
    const int64_t units = (int64_t)a0.R * a0.n_layers * a0.H;
    if (units == 0) return cudaSuccess;
    ChainArgs c = a0;   // the state of the group from a zero start
    c.S_init = nullptr;
    c.op = 0;
    cudaError_t e = launch_compose_chain(c, s);
    if (e != cudaSuccess) return e;
    if (a0.fam == HYPIC_DENSE) {   // the operator chain M_pn ... M_p1
        ChainArgs o = a0;
        o.op = 1;
        o.S_init = nullptr;
        o.dv = o.dk;
        o.pool_S = a0.pool_M;   // never read in operator mode; shaped like the operator
        o.S_out = M_out;
        o.lam_out = lam_out;
        e = chain_dense_tc_supported(o) ? launch_chain_dense_tc(o, s) : dispatch_dd<DenseChainF>(o, s, o.dk, o.dk);
        if (e != cudaSuccess) return e;
        prefix_finish_kernel<true, false><<<(unsigned)units, 256, 0, s>>>(a0, lam_out, M_out);
    } else if (a0.fam == HYPIC_DIAG) {
        prefix_finish_kernel<false, true><<<(unsigned)units, 256, 0, s>>>(a0, lam_out, nullptr);
    } else {
        prefix_finish_kernel<false, false><<<(unsigned)units, 256, 0, s>>>(a0, lam_out, nullptr);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- two-level tree
//
// With few (request, layer, head) units a chain runs on few SMs, one pool entry
// after another.  The operator of a concatenation is the product of the operators,
// T(C1.C2) = T(C2) T(C1), so any run of consecutive entries can first be folded into
// one cached pair.  Level 1 folds groups of gs entries of every chain in parallel
// (the composed-prefix kernels, one virtual request per (request, group)); level 2
// folds each request's group pairs in order into S_init (the chain kernels).

namespace {

constexpr int kTreeMinChain = 8;   // shorter chains gain nothing from a second level

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
        n = 148;
    return n;
}

int64_t up256(int64_t b) { return (b + 255) / 256 * 256; }

struct TreeLayout {
    int G;                       // groups per request
    int64_t lam, M, S, si1, cl1, si2, cl2, total;   // byte offsets
};

TreeLayout tree_layout(const ChainArgs &a, int gs) {
    TreeLayout t{};
    t.G = (a.max_chain + gs - 1) / gs;
    const int64_t entries = (int64_t)a.R * t.G * a.n_layers * a.H;
    const int nl = a.fam == HYPIC_DIAG ? a.dk : 1;
    int64_t o = 0;
    t.lam = o;
    o += up256(entries * nl * 4);
    t.M = o;
    if (a.fam == HYPIC_DENSE) o += up256(entries * a.dk * a.dk * 4);
    t.S = o;
    o += up256(entries * a.dk * a.dv * 4);
    t.si1 = o;
    o += up256((int64_t)a.R * t.G * gs * 4);
    t.cl1 = o;
    o += up256((int64_t)a.R * t.G * 4);
    t.si2 = o;
    o += up256((int64_t)a.R * t.G * 4);
    t.cl2 = o;
    o += up256((int64_t)a.R * 4);
    t.total = o;
    return t;
}

// one thread per (request, group): the group's entries and length (level 1), the
// request's group list and count (level 2); a chain length outside [0, max_chain]
// is clamped and reported like the chain kernels do
__global__ void tree_index_kernel(const ChainArgs a, int gs, int G, int32_t *si1, int32_t *cl1, int32_t *si2,
                                  int32_t *cl2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)a.R * G) return;
    const int r = (int)(i / G), g = (int)(i % G);
    int n = a.chain_len[r];
    if (n < 0 || n > a.max_chain) {
        if (g == 0) flag_index_error(a.d_err);
        n = n < 0 ? 0 : a.max_chain;
    }
    const int rem = n - g * gs;
    cl1[i] = rem <= 0 ? 0 : (rem < gs ? rem : gs);
    for (int j = 0; j < gs; ++j) {
        const int c = g * gs + j;
        si1[i * gs + j] = c < a.max_chain ? a.seg_idx[(int64_t)r * a.max_chain + c] : 0;
    }
    si2[i] = (int32_t)i;
    if (g == 0) cl2[r] = (n + gs - 1) / gs;
}

}  // namespace

int tree_group_size(const ChainArgs &a) {
    const int64_t units = (int64_t)a.R * a.n_layers * a.H;
    const int sms = sm_count();
    if (a.max_chain < kTreeMinChain || units >= 2 * (int64_t)sms) return 0;
    // about four CTAs per SM in level 1, at least 4 entries a group
    const int64_t want_groups = (4 * (int64_t)sms + units - 1) / units;
    int gs = (int)((a.max_chain + want_groups - 1) / want_groups);
    if (gs < 4) gs = 4;
    return gs >= a.max_chain ? 0 : gs;
}

int64_t tree_bytes(const ChainArgs &a, int gs) { return gs > 0 ? tree_layout(a, gs).total : 0; }

cudaError_t launch_compose_chain_tree(const ChainArgs &a, int gs, void *ws, cudaStream_t s) {
    const TreeLayout t = tree_layout(a, gs);
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *si1 = reinterpret_cast<int32_t *>(w + t.si1), *cl1 = reinterpret_cast<int32_t *>(w + t.cl1);
    int32_t *si2 = reinterpret_cast<int32_t *>(w + t.si2), *cl2 = reinterpret_cast<int32_t *>(w + t.cl2);
    const int64_t groups = (int64_t)a.R * t.G;
    tree_index_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(a, gs, t.G, si1, cl1, si2, cl2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // level 1: every group's pair (a composed prefix per virtual request)
    ChainArgs l1 = a;
    l1.R = (int)groups;
    l1.max_chain = gs;
    l1.chain_len = cl1;
    l1.seg_idx = si1;
    l1.S_init = nullptr;
    l1.S_out = reinterpret_cast<float *>(w + t.S);
    float *lam1 = reinterpret_cast<float *>(w + t.lam);
    float *M1 = a.fam == HYPIC_DENSE ? reinterpret_cast<float *>(w + t.M) : nullptr;
    e = launch_compose_prefix(l1, lam1, M1, s);
    if (e != cudaSuccess) return e;
    // level 2: each request folds its groups' pairs in order
    ChainArgs l2 = a;
    l2.max_chain = t.G;
    l2.chain_len = cl2;
    l2.seg_idx = si2;
    l2.P = (int)groups;
    l2.pool_lam = lam1;
    l2.pool_M = M1;
    l2.pool_S = l1.S_out;
    return launch_compose_chain(l2, s);
}

cudaError_t launch_compose_chain(const ChainArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.R * a.n_layers * a.H;
    if (units == 0) return cudaSuccess;
    if (chain_dense_tc_supported(a)) return launch_chain_dense_tc(a, s);
    if (a.fam == HYPIC_DENSE) return dispatch_dd<DenseChainF>(a, s, a.dk, a.dv);
    if (a.fam == HYPIC_DIAG)
        chain_sd_kernel<true><<<(unsigned)units, 256, 0, s>>>(a);
    else
        chain_sd_kernel<false><<<(unsigned)units, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hypic
