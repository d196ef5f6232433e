// internal.cuh -- declarations shared by the translation units of libhypic.
// Launchers return a cudaError_t; api.cu turns that into a hypic_status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/hypic.h"

namespace hypic {

struct ScanArgs {
    int fam;          // hypic_family
    int in_dtype;     // hypic_dtype
    int n_layers, n_seg, H, dk, dv;
    int64_t N;        // tokens per layer
    const int64_t *seg_offsets;
    const void *q, *k, *v;
    const float *alpha, *beta;
    float *lam_out, *M_out, *S_out;
    void *o_out;
    float *ws;        // caller-owned scratch of the two-pass dense scan (or NULL)
    int *d_err;
    const int *order = nullptr;   // two-pass dense: segments longest first (or NULL: as given)
    // token-by-token kernel: only the units unit_list[0 .. *unit_count) (device; or NULL: all)
    const int *unit_list = nullptr, *unit_count = nullptr;
};

struct ComposeArgs {
    int fam, n, H, dk, dv;
    const float *lam, *M, *S_prev, *S_C;
    float *S_out;
    const float *lam_prev, *M_prev;
    float *lam_out, *M_out;
};

struct ChainArgs {
    int fam, R, n_layers, H, dk, dv, max_chain, P;
    const int32_t *chain_len, *seg_idx;
    // without seg_idx: the entries of request r are seg_first[r], seg_first[r] + 1, ... (or NULL)
    const int32_t *seg_first = nullptr;
    const float *pool_lam, *pool_M, *pool_S, *S_init;
    float *S_out;
    int *d_err;
    // operator mode (dense, kda): S_out <- M_pn ... M_p1 from I (no S_p, no exp(lambda)),
    // rescaled by powers of two on the way; the exponent per unit goes to lam_out
    int op = 0;
    float *lam_out = nullptr;
    // dense tensor-core chains: bf16 hi / lo operands (three products a step) instead of
    // hi / mid / lo (six); for chains inside a scan of bf16 inputs (1e-3), not the fp32 compose
    int two_way = 0;
};

// cuTensorMapEncodeTiled through the runtime's driver entry point (nullptr if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// 3-D tiled map over a [rows][mid][inner] array (element size esize) with box {box0, 1, box2}.
bool make_tensor_map_3d(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner,
                        uint64_t mid, uint64_t rows, uint32_t box0, uint32_t box2, CUtensorMapSwizzle sw);

// Token-by-token fp32 recurrence on CUDA cores, every family, optional o_t.
cudaError_t launch_scan_recurrent(const ScanArgs &a, cudaStream_t s);

// Scalar / diagonal scan on tcgen05 tensor cores (bf16 inputs, d_k = d_v = 128, no o_t).
bool scan_sd_tc_supported(const ScanArgs &a);
cudaError_t launch_scan_sd_tc(const ScanArgs &a, cudaStream_t s);
bool scan_sd_bal_shape(const ScanArgs &a);        // the balanced schedule (scratch) takes it
int64_t scan_sd_bal_bytes();                      // its scratch
cudaError_t launch_scan_sd_bal(const ScanArgs &a, cudaStream_t s);
// Scalar gates with the per-token outputs o_t, chunks in order on tcgen05 (bf16, 128 x 128).
bool scan_sd_o_supported(const ScanArgs &a);
cudaError_t launch_scan_sd_o(const ScanArgs &a, cudaStream_t s);
// Diagonal gates with o_t, chunks in order on tcgen05 (bf16, 128 x 128).
bool scan_diag_o_supported(const ScanArgs &a);
cudaError_t launch_scan_diag_o(const ScanArgs &a, cudaStream_t s);

// Gated delta rule scan on tcgen05 tensor cores (bf16 inputs, d_k = d_v = 128, no o_t).
bool scan_dense_tc_supported(const ScanArgs &a);
cudaError_t launch_scan_dense_tc(const ScanArgs &a, cudaStream_t s);
bool scan_dense_ws_shape(const ScanArgs &a);       // sizes / options the two-pass form takes
bool scan_dense_ws_supported(const ScanArgs &a);   // ... and the runtime can encode its tensor maps
int64_t scan_dense_ws_bytes(const ScanArgs &a);
cudaError_t launch_scan_dense_ws(const ScanArgs &a, cudaStream_t s);
// KDA-style gates on tcgen05 (bf16, 128 x 128, no o_t): each chunk's pair in parallel,
// then the composed-prefix kernels over each segment's chunks.  Scratch-backed.
constexpr int64_t kKdaMaxScratch = (int64_t)64 << 30;   // beyond this the token-by-token kernel
bool scan_kda_tc_shape(const ScanArgs &a);
bool scan_kda_tc_supported(const ScanArgs &a);
int64_t scan_kda_tc_bytes(const ScanArgs &a);
cudaError_t launch_scan_kda_tc(const ScanArgs &a, cudaStream_t s);
int64_t static_scratch_bytes();            // size of the fixed scratch of hypic_segment_scan_static
cudaError_t static_scratch(void **p);      // its address on the current device

// Dense chained composition on tcgen05 (bf16 three-way splits, fp32 state), d_k = d_v = 128.
bool chain_dense_tc_supported(const ChainArgs &a);
cudaError_t launch_chain_dense_tc(const ChainArgs &a, cudaStream_t s);

cudaError_t launch_compose(const ComposeArgs &a, cudaStream_t s);
cudaError_t launch_compose_chain(const ChainArgs &a, cudaStream_t s);
// The cached pair of each request's ordered pool entries: S from a zero state into
// a.S_out, T = T_pn ... T_p1 into lam_out (and M_out for dense, kda).
cudaError_t launch_compose_prefix(const ChainArgs &a, float *lam_out, float *M_out, cudaStream_t s);
// Two-level tree for few (request, layer, head) units with long chains: groups of
// `gs` consecutive entries fold in parallel into cached pairs (composed prefixes),
// then each unit folds its groups' pairs in order.  tree_group_size() is 0 where the
// plain chain is used; tree_bytes() is the scratch the tree needs.
int tree_group_size(const ChainArgs &a);
int64_t tree_bytes(const ChainArgs &a, int gs);
cudaError_t launch_compose_chain_tree(const ChainArgs &a, int gs, void *ws, cudaStream_t s);

// Seam-window advance, then the composition of the rest of the segment.
struct SeamArgs {
    int fam, in_dtype, n, w, H, dk, dv;
    const void *q, *k, *v;
    const float *alpha, *beta;
    const float *lam, *M, *S_prev, *S_C;
    float *S_out;
    void *o_out;
};
cudaError_t launch_seam_compose(const SeamArgs &a, cudaStream_t s);

// Report a device-side index problem without trapping.
__device__ __forceinline__ void flag_index_error(int *d_err) {
    if (d_err) atomicExch(d_err, (int)HYPIC_EINDEX);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

}  // namespace hypic
