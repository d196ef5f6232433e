// api.cu -- the extern "C" entry points of libhypic: argument checks on the
// host, then one or more launches on the caller's stream.  No allocation, no
// global state, no synchronisation.
#include <stdint.h>

#include <mutex>

#include "internal.cuh"

namespace hypic {

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_tensor_map_3d(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner,
                        uint64_t mid, uint64_t rows, uint32_t box0, uint32_t box2, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {inner, mid, rows};
    const cuuint64_t strides[2] = {inner * esize, inner * mid * esize};
    const cuuint32_t box[3] = {box0, 1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace hypic

namespace {

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool head_size_ok(int d) { return d == 32 || d == 64 || d == 128; }

bool family_ok(int fam) { return fam >= HYPIC_SCALAR && fam <= HYPIC_KDA; }
bool has_m(int fam) { return fam == HYPIC_DENSE || fam == HYPIC_KDA; }        // operator exp(lambda) M
bool gate_per_channel(int fam) { return fam == HYPIC_DIAG || fam == HYPIC_KDA; }
// the composition of a KDA pair is that of a dense pair: both are (lambda, M)
int compose_family(int fam) { return fam == HYPIC_KDA ? HYPIC_DENSE : fam; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? HYPIC_OK : HYPIC_ECUDA; }

}  // namespace

extern "C" {

int hypic_version(void) { return 100; }

const char *hypic_status_string(int status) {
    switch (status) {
        case HYPIC_OK: return "ok";
        case HYPIC_EINVAL: return "invalid argument";
        case HYPIC_EUNSUPPORTED: return "unsupported size or option";
        case HYPIC_EALIGN: return "misaligned pointer";
        case HYPIC_ECUDA: return "CUDA error";
        case HYPIC_EINDEX: return "index out of range (device side)";
        case HYPIC_ETIMEOUT: return "a device-side wait timed out";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

// Host checks shared by hypic_segment_scan and hypic_segment_scan_ws; fills `a`.
// Returns HYPIC_OK and sets *nothing_to_do when there is no work.
int scan_args(int fam, int in_dtype, int n_layers, int n_seg, int64_t total_tokens, int n_heads, int d_k,
              int d_v, const int64_t *seg_offsets, const void *q, const void *k, const void *v,
              const float *alpha, const float *beta, float *lam_out, float *M_out, float *S_out, void *o_out,
              int *d_err, hypic::ScanArgs &a, bool &nothing_to_do) {
    nothing_to_do = false;
    if (!family_ok(fam)) return HYPIC_EINVAL;
    if (in_dtype != HYPIC_BF16 && in_dtype != HYPIC_F32) return HYPIC_EINVAL;
    if (n_layers < 0 || n_seg < 0 || total_tokens < 0 || n_heads <= 0) return HYPIC_EINVAL;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n_layers * n_seg * n_heads > INT32_MAX) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n_layers * total_tokens * n_heads > (INT64_MAX / 256)) return HYPIC_EUNSUPPORTED;
    if (n_layers == 0 || n_seg == 0) {
        nothing_to_do = true;
        return HYPIC_OK;
    }
    const bool has_tokens = total_tokens > 0;
    if (!seg_offsets || !lam_out || !S_out) return HYPIC_EINVAL;
    if (has_tokens && (!k || !v || !alpha)) return HYPIC_EINVAL;
    if (has_m(fam) != (M_out != nullptr)) return HYPIC_EINVAL;
    if (o_out && !q && has_tokens) return HYPIC_EINVAL;
    if (!aligned(seg_offsets, 8)) return HYPIC_EALIGN;
    const void *a16[] = {q, k, v, o_out, S_out, M_out, gate_per_channel(fam) ? alpha : nullptr,
                         fam == HYPIC_DIAG ? lam_out : nullptr};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return HYPIC_EALIGN;
    const void *a4[] = {alpha, beta, lam_out, d_err};
    for (const void *p : a4)
        if (p && !aligned(p, 4)) return HYPIC_EALIGN;

    a.fam = fam;
    a.in_dtype = in_dtype;
    a.n_layers = n_layers;
    a.n_seg = n_seg;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.N = total_tokens;
    a.seg_offsets = seg_offsets;
    a.q = o_out ? q : nullptr;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.lam_out = lam_out;
    a.M_out = M_out;
    a.S_out = S_out;
    a.o_out = o_out;
    a.d_err = d_err;
    a.ws = nullptr;
    return HYPIC_OK;
}

}  // namespace

extern "C" {

int hypic_segment_scan(int fam, int in_dtype, int n_layers, int n_seg, int64_t total_tokens,
                       int n_heads, int d_k, int d_v, const int64_t *seg_offsets, const void *q,
                       const void *k, const void *v, const float *alpha, const float *beta,
                       float *lam_out, float *M_out, float *S_out, void *o_out, int *d_err,
                       void *cuda_stream) {
    hypic::ScanArgs a;
    bool none;
    const int rc = scan_args(fam, in_dtype, n_layers, n_seg, total_tokens, n_heads, d_k, d_v, seg_offsets, q, k,
                             v, alpha, beta, lam_out, M_out, S_out, o_out, d_err, a, none);
    if (rc != HYPIC_OK || none) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (hypic::scan_sd_o_supported(a)) return from_cuda(hypic::launch_scan_sd_o(a, s));
    if (hypic::scan_diag_o_supported(a)) return from_cuda(hypic::launch_scan_diag_o(a, s));
    if (hypic::scan_sd_tc_supported(a)) return from_cuda(hypic::launch_scan_sd_tc(a, s));
    if (hypic::scan_dense_tc_supported(a)) return from_cuda(hypic::launch_scan_dense_tc(a, s));
    return from_cuda(hypic::launch_scan_recurrent(a, s));
}

int64_t hypic_segment_scan_workspace_bytes(int fam, int in_dtype, int n_layers, int n_seg,
                                           int64_t total_tokens, int n_heads, int d_k, int d_v,
                                           int with_o) {
    if (!family_ok(fam) || n_layers < 0 || n_seg < 0 || total_tokens < 0 || n_heads <= 0) return HYPIC_EINVAL;
    hypic::ScanArgs a{};
    a.fam = fam;
    a.in_dtype = in_dtype;
    a.n_layers = n_layers;
    a.n_seg = n_seg;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.N = total_tokens;
    a.o_out = with_o ? reinterpret_cast<void *>(16) : nullptr;   // only tested against NULL
    if (n_layers == 0 || n_seg == 0) return 0;
    if (hypic::scan_dense_ws_shape(a)) return hypic::scan_dense_ws_bytes(a);
    if (hypic::scan_kda_tc_shape(a)) return hypic::scan_kda_tc_bytes(a);
    if (hypic::scan_sd_bal_shape(a)) return hypic::scan_sd_bal_bytes();
    return 0;
}

int hypic_segment_scan_ws(int fam, int in_dtype, int n_layers, int n_seg, int64_t total_tokens,
                          int n_heads, int d_k, int d_v, const int64_t *seg_offsets, const void *q,
                          const void *k, const void *v, const float *alpha, const float *beta,
                          float *lam_out, float *M_out, float *S_out, void *o_out, void *workspace,
                          int64_t workspace_bytes, int *d_err, void *cuda_stream) {
    hypic::ScanArgs a;
    bool none;
    const int rc = scan_args(fam, in_dtype, n_layers, n_seg, total_tokens, n_heads, d_k, d_v, seg_offsets, q, k,
                             v, alpha, beta, lam_out, M_out, S_out, o_out, d_err, a, none);
    if (rc != HYPIC_OK || none) return rc;
    if (workspace_bytes < 0) return HYPIC_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (hypic::scan_dense_ws_shape(a)) {
        if (!workspace || workspace_bytes < hypic::scan_dense_ws_bytes(a)) return HYPIC_EINVAL;
        if (!aligned(workspace, 256)) return HYPIC_EALIGN;
    }
    if (hypic::scan_dense_ws_supported(a)) {
        a.ws = static_cast<float *>(workspace);
        return from_cuda(hypic::launch_scan_dense_ws(a, s));
    }
    if (hypic::scan_kda_tc_shape(a)) {
        if (!workspace || workspace_bytes < hypic::scan_kda_tc_bytes(a)) return HYPIC_EINVAL;
        if (!aligned(workspace, 256)) return HYPIC_EALIGN;
        if (hypic::scan_kda_tc_supported(a)) {
            a.ws = static_cast<float *>(workspace);
            return from_cuda(hypic::launch_scan_kda_tc(a, s));
        }
    }
    if (hypic::scan_sd_bal_shape(a) && hypic::scan_sd_tc_supported(a)) {
        if (!workspace || workspace_bytes < hypic::scan_sd_bal_bytes()) return HYPIC_EINVAL;
        if (!aligned(workspace, 256)) return HYPIC_EALIGN;
        a.ws = static_cast<float *>(workspace);
        return from_cuda(hypic::launch_scan_sd_bal(a, s));
    }
    if (hypic::scan_sd_o_supported(a)) return from_cuda(hypic::launch_scan_sd_o(a, s));
    if (hypic::scan_diag_o_supported(a)) return from_cuda(hypic::launch_scan_diag_o(a, s));
    if (hypic::scan_sd_tc_supported(a)) return from_cuda(hypic::launch_scan_sd_tc(a, s));
    if (hypic::scan_dense_tc_supported(a)) return from_cuda(hypic::launch_scan_dense_tc(a, s));
    return from_cuda(hypic::launch_scan_recurrent(a, s));
}

int hypic_segment_scan_static(int fam, int in_dtype, int n_layers, int n_seg, int64_t total_tokens,
                              int n_heads, int d_k, int d_v, const int64_t *seg_offsets, const void *k,
                              const void *v, const float *alpha, const float *beta, float *lam_out,
                              float *M_out, float *S_out, int *d_err, void *cuda_stream) {
    hypic::ScanArgs a;
    bool none;
    const int rc = scan_args(fam, in_dtype, n_layers, n_seg, total_tokens, n_heads, d_k, d_v, seg_offsets,
                             nullptr, k, v, alpha, beta, lam_out, M_out, S_out, nullptr, d_err, a, none);
    if (rc != HYPIC_OK || none) return rc;
    if (fam != HYPIC_DENSE || in_dtype != HYPIC_BF16 || d_k != 128 || d_v != 128) return HYPIC_EUNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (total_tokens == 0) {   // only empty segments: lambda = 0, M = I, S = 0, written without scratch
        if (hypic::scan_dense_tc_supported(a)) return from_cuda(hypic::launch_scan_dense_tc(a, s));
        return from_cuda(hypic::launch_scan_recurrent(a, s));
    }
    if (!hypic::scan_dense_ws_shape(a)) return HYPIC_EUNSUPPORTED;
    if (hypic::scan_dense_ws_bytes(a) > hypic::static_scratch_bytes()) return HYPIC_EUNSUPPORTED;
    if (!hypic::scan_dense_ws_supported(a)) return HYPIC_ECUDA;
    void *scratch = nullptr;
    if (hypic::static_scratch(&scratch) != cudaSuccess || !scratch) return HYPIC_ECUDA;
    a.ws = static_cast<float *>(scratch);
    return from_cuda(hypic::launch_scan_dense_ws(a, s));
}

int hypic_compose(int fam, int n, int n_heads, int d_k, int d_v, const float *lam, const float *M,
                  const float *S_prev, const float *S_C, float *S_out, const float *lam_prev,
                  const float *M_prev, float *lam_out, float *M_out, void *cuda_stream) {
    if (!family_ok(fam)) return HYPIC_EINVAL;
    if (n < 0 || n_heads <= 0) return HYPIC_EINVAL;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n * n_heads > INT32_MAX) return HYPIC_EUNSUPPORTED;
    if (n == 0) return HYPIC_OK;
    if (!lam || !S_C || !S_out) return HYPIC_EINVAL;
    if (has_m(fam) != (M != nullptr)) return HYPIC_EINVAL;
    if ((lam_prev == nullptr) != (lam_out == nullptr)) return HYPIC_EINVAL;
    if (has_m(fam)) {
        if ((M_prev == nullptr) != (lam_out == nullptr) || (M_out == nullptr) != (lam_out == nullptr))
            return HYPIC_EINVAL;
    } else if (M_prev || M_out) {
        return HYPIC_EINVAL;
    }
    const void *a16[] = {M, S_prev, S_C, S_out, M_prev, M_out,
                         fam == HYPIC_DIAG ? lam : nullptr, fam == HYPIC_DIAG ? lam_prev : nullptr,
                         fam == HYPIC_DIAG ? lam_out : nullptr};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return HYPIC_EALIGN;
    const void *a4[] = {lam, lam_prev, lam_out};
    for (const void *p : a4)
        if (p && !aligned(p, 4)) return HYPIC_EALIGN;
    // S_out may be S_prev; any other overlap with an input is not supported
    const size_t sbytes = (size_t)n * n_heads * d_k * d_v * sizeof(float);
    const size_t mbytes = (size_t)n * n_heads * d_k * d_k * sizeof(float);
    auto overlaps = [](const void *x, size_t xb, const void *y, size_t yb) {
        if (!x || !y) return false;
        const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(y);
        return a < b + yb && b < a + xb;
    };
    if (S_out != S_C && overlaps(S_out, sbytes, S_C, sbytes)) return HYPIC_EINVAL;
    if (S_prev && S_out != S_prev && overlaps(S_out, sbytes, S_prev, sbytes)) return HYPIC_EINVAL;
    if (has_m(fam) &&
        (overlaps(S_out, sbytes, M, mbytes) || overlaps(S_out, sbytes, M_prev, mbytes) ||
         overlaps(M_out, mbytes, M, mbytes) || overlaps(M_out, mbytes, M_prev, mbytes)))
        return HYPIC_EINVAL;
    // lam_out is written while other threads (or another part of the grid) still
    // read lam and lam_prev, so it may alias neither
    const size_t lbytes = (size_t)n * n_heads * (fam == HYPIC_DIAG ? d_k : 1) * sizeof(float);
    if (overlaps(lam_out, lbytes, lam, lbytes) || overlaps(lam_out, lbytes, lam_prev, lbytes) ||
        overlaps(lam_out, lbytes, S_out, sbytes) || overlaps(lam_out, lbytes, M_out, mbytes))
        return HYPIC_EINVAL;

    hypic::ComposeArgs a;
    a.fam = compose_family(fam);
    a.n = n;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.lam = lam;
    a.M = M;
    a.S_prev = S_prev;
    a.S_C = S_C;
    a.S_out = S_out;
    a.lam_prev = lam_prev;
    a.M_prev = M_prev;
    a.lam_out = lam_out;
    a.M_out = M_out;
    return from_cuda(hypic::launch_compose(a, static_cast<cudaStream_t>(cuda_stream)));
}

int hypic_seam_compose(int fam, int in_dtype, int n, int w, int n_heads, int d_k, int d_v, const void *q,
                       const void *k, const void *v, const float *alpha, const float *beta, const float *lam,
                       const float *M, const float *S_prev, const float *S_C, float *S_out, void *o_out,
                       void *cuda_stream) {
    if (!family_ok(fam)) return HYPIC_EINVAL;
    if (in_dtype != HYPIC_BF16 && in_dtype != HYPIC_F32) return HYPIC_EINVAL;
    if (n < 0 || n_heads <= 0 || w < 0) return HYPIC_EINVAL;
    if (w > 4096) return HYPIC_EUNSUPPORTED;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n * n_heads * (d_v / 32) > INT32_MAX) return HYPIC_EUNSUPPORTED;   // one CTA per 32 columns
    if (n == 0) return HYPIC_OK;
    if (!lam || !S_C || !S_out) return HYPIC_EINVAL;
    if (has_m(fam) != (M != nullptr)) return HYPIC_EINVAL;
    if (w > 0 && (!k || !v || !alpha || (o_out && !q))) return HYPIC_EINVAL;
    const void *a16[] = {M, S_prev, S_C, S_out, fam == HYPIC_DIAG ? lam : nullptr};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return HYPIC_EALIGN;
    const void *a4[] = {lam, alpha, beta};
    for (const void *p : a4)
        if (p && !aligned(p, 4)) return HYPIC_EALIGN;
    const uintptr_t ea = in_dtype == HYPIC_BF16 ? 2 : 4;
    const void *ae[] = {q, k, v, o_out};
    for (const void *p : ae)
        if (p && !aligned(p, ea)) return HYPIC_EALIGN;
    const size_t sbytes = (size_t)n * n_heads * d_k * d_v * sizeof(float);
    const size_t mbytes = (size_t)n * n_heads * d_k * d_k * sizeof(float);
    const size_t es = in_dtype == HYPIC_BF16 ? 2 : 4;
    const size_t obytes = (size_t)n * w * n_heads * d_v * es;
    auto overlaps = [](const void *x, size_t xb, const void *y, size_t yb) {
        if (!x || !y) return false;
        const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(y);
        return a < b + yb && b < a + xb;
    };
    if (overlaps(S_out, sbytes, S_C, sbytes) || overlaps(S_out, sbytes, M, mbytes)) return HYPIC_EINVAL;
    if (S_prev && S_out != S_prev && overlaps(S_out, sbytes, S_prev, sbytes)) return HYPIC_EINVAL;
    if (o_out && (overlaps(o_out, obytes, S_out, sbytes) || overlaps(o_out, obytes, S_prev, sbytes) ||
                  overlaps(o_out, obytes, q, (size_t)n * w * n_heads * d_k * es) ||
                  overlaps(o_out, obytes, k, (size_t)n * w * n_heads * d_k * es) ||
                  overlaps(o_out, obytes, v, obytes)))
        return HYPIC_EINVAL;

    hypic::SeamArgs a;
    a.fam = fam;
    a.in_dtype = in_dtype;
    a.n = n;
    a.w = w;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.q = o_out ? q : nullptr;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.lam = lam;
    a.M = M;
    a.S_prev = S_prev;
    a.S_C = S_C;
    a.S_out = S_out;
    a.o_out = w > 0 ? o_out : nullptr;
    return from_cuda(hypic::launch_seam_compose(a, static_cast<cudaStream_t>(cuda_stream)));
}

}  // extern "C"

namespace {

// Host checks of hypic_compose_chain(_ws); fills `a`.  Returns HYPIC_OK and sets
// *nothing_to_do when there is no work.
int chain_args(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v, int max_chain,
               const int32_t *chain_len, const int32_t *seg_idx, int pool_size, const float *pool_lam,
               const float *pool_M, const float *pool_S, const float *S_init, float *S_out, int *d_err,
               hypic::ChainArgs &a, bool &nothing_to_do) {
    nothing_to_do = false;
    if (!family_ok(fam)) return HYPIC_EINVAL;
    if (n_req < 0 || n_layers < 0 || n_heads <= 0 || max_chain < 0 || pool_size < 0)
        return HYPIC_EINVAL;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n_req * n_layers * n_heads > INT32_MAX) return HYPIC_EUNSUPPORTED;
    if (n_req == 0 || n_layers == 0) {
        nothing_to_do = true;
        return HYPIC_OK;
    }
    if (!chain_len || !S_out) return HYPIC_EINVAL;
    if (max_chain > 0 && (!seg_idx || pool_size == 0 || !pool_lam || !pool_S)) return HYPIC_EINVAL;
    if (max_chain > 0 && has_m(fam) != (pool_M != nullptr)) return HYPIC_EINVAL;
    const void *a16[] = {pool_M, pool_S, S_init, S_out, fam == HYPIC_DIAG ? pool_lam : nullptr};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return HYPIC_EALIGN;
    const void *a4[] = {chain_len, seg_idx, pool_lam, d_err};
    for (const void *p : a4)
        if (p && !aligned(p, 4)) return HYPIC_EALIGN;
    // S_out is written while other chains still read the pool: no overlap with it
    // (S_out may be S_init itself, each chain reading its own state before writing it)
    {
        const int64_t units = (int64_t)n_req * n_layers * n_heads;
        const int64_t entries = (int64_t)pool_size * n_layers * n_heads;
        const int nl = fam == HYPIC_DIAG ? d_k : 1;
        auto overlaps = [](const void *x, size_t xb, const void *y, size_t yb) {
            if (!x || !y) return false;
            const char *p = static_cast<const char *>(x), *q = static_cast<const char *>(y);
            return p < q + yb && q < p + xb;
        };
        const size_t sb = (size_t)units * d_k * d_v * 4;
        if (overlaps(S_out, sb, pool_S, (size_t)entries * d_k * d_v * 4) ||
            overlaps(S_out, sb, pool_M, (size_t)entries * d_k * d_k * 4) ||
            overlaps(S_out, sb, pool_lam, (size_t)entries * nl * 4) ||
            (S_init && S_init != S_out && overlaps(S_out, sb, S_init, sb)))
            return HYPIC_EINVAL;
    }

    a.fam = compose_family(fam);
    a.R = n_req;
    a.n_layers = n_layers;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.max_chain = max_chain;
    a.P = pool_size;
    a.chain_len = chain_len;
    a.seg_idx = seg_idx;
    a.pool_lam = pool_lam;
    a.pool_M = pool_M;
    a.pool_S = pool_S;
    a.S_init = S_init;
    a.S_out = S_out;
    a.d_err = d_err;
    return HYPIC_OK;
}

}  // namespace

extern "C" {

int hypic_compose_chain(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v,
                        int max_chain, const int32_t *chain_len, const int32_t *seg_idx,
                        int pool_size, const float *pool_lam, const float *pool_M,
                        const float *pool_S, const float *S_init, float *S_out, int *d_err,
                        void *cuda_stream) {
    hypic::ChainArgs a;
    bool none;
    const int rc = chain_args(fam, n_req, n_layers, n_heads, d_k, d_v, max_chain, chain_len, seg_idx, pool_size,
                              pool_lam, pool_M, pool_S, S_init, S_out, d_err, a, none);
    if (rc != HYPIC_OK || none) return rc;
    return from_cuda(hypic::launch_compose_chain(a, static_cast<cudaStream_t>(cuda_stream)));
}

int64_t hypic_compose_chain_workspace_bytes(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v,
                                            int max_chain) {
    if (!family_ok(fam) || n_req < 0 || n_layers < 0 || n_heads <= 0 || max_chain < 0) return HYPIC_EINVAL;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if (n_req == 0 || n_layers == 0) return 0;
    hypic::ChainArgs a{};
    a.fam = compose_family(fam);
    a.R = n_req;
    a.n_layers = n_layers;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.max_chain = max_chain;
    return hypic::tree_bytes(a, hypic::tree_group_size(a));
}

int hypic_compose_chain_ws(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v, int max_chain,
                           const int32_t *chain_len, const int32_t *seg_idx, int pool_size,
                           const float *pool_lam, const float *pool_M, const float *pool_S,
                           const float *S_init, float *S_out, void *workspace, int64_t workspace_bytes,
                           int *d_err, void *cuda_stream) {
    hypic::ChainArgs a;
    bool none;
    const int rc = chain_args(fam, n_req, n_layers, n_heads, d_k, d_v, max_chain, chain_len, seg_idx, pool_size,
                              pool_lam, pool_M, pool_S, S_init, S_out, d_err, a, none);
    if (rc != HYPIC_OK || none) return rc;
    if (workspace_bytes < 0) return HYPIC_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int gs = hypic::tree_group_size(a);
    if (gs == 0) return from_cuda(hypic::launch_compose_chain(a, s));
    const int64_t need = hypic::tree_bytes(a, gs);
    if (!workspace || workspace_bytes < need) return HYPIC_EINVAL;
    if (!aligned(workspace, 256)) return HYPIC_EALIGN;
    // the scratch may overlap neither the pool nor the states
    const int64_t units = (int64_t)n_req * n_layers * n_heads;
    const int64_t entries = (int64_t)pool_size * n_layers * n_heads;
    const char *w = static_cast<const char *>(workspace);
    auto hits = [&](const void *p, size_t b) {
        const char *q = static_cast<const char *>(p);
        return p && q < w + need && w < q + b;
    };
    if (hits(pool_S, (size_t)entries * d_k * d_v * 4) || hits(pool_M, (size_t)entries * d_k * d_k * 4) ||
        hits(pool_lam, (size_t)entries * d_k * 4) || hits(S_out, (size_t)units * d_k * d_v * 4) ||
        hits(S_init, (size_t)units * d_k * d_v * 4) || hits(chain_len, (size_t)n_req * 4) ||
        hits(seg_idx, (size_t)n_req * max_chain * 4))
        return HYPIC_EINVAL;
    return from_cuda(hypic::launch_compose_chain_tree(a, gs, workspace, s));
}

int hypic_compose_prefix(int fam, int n_req, int n_layers, int n_heads, int d_k, int d_v, int max_chain,
                         const int32_t *chain_len, const int32_t *seg_idx, int pool_size, const float *pool_lam,
                         const float *pool_M, const float *pool_S, float *lam_out, float *M_out, float *S_out,
                         int *d_err, void *cuda_stream) {
    if (!family_ok(fam)) return HYPIC_EINVAL;
    if (n_req < 0 || n_layers < 0 || n_heads <= 0 || max_chain < 0 || pool_size < 0) return HYPIC_EINVAL;
    if (!head_size_ok(d_k) || !head_size_ok(d_v)) return HYPIC_EUNSUPPORTED;
    if ((int64_t)n_req * n_layers * n_heads > INT32_MAX) return HYPIC_EUNSUPPORTED;
    if (n_req == 0 || n_layers == 0) return HYPIC_OK;
    if (!chain_len || !S_out || !lam_out) return HYPIC_EINVAL;
    if (has_m(fam) != (M_out != nullptr)) return HYPIC_EINVAL;
    if (max_chain > 0 && (!seg_idx || pool_size == 0 || !pool_lam || !pool_S)) return HYPIC_EINVAL;
    if (max_chain > 0 && has_m(fam) != (pool_M != nullptr)) return HYPIC_EINVAL;
    const void *a16[] = {pool_M, pool_S, M_out, S_out, fam == HYPIC_DIAG ? pool_lam : nullptr,
                         fam == HYPIC_DIAG ? lam_out : nullptr};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return HYPIC_EALIGN;
    const void *a4[] = {chain_len, seg_idx, pool_lam, lam_out, d_err};
    for (const void *p : a4)
        if (p && !aligned(p, 4)) return HYPIC_EALIGN;
    // the outputs overlap neither one another nor the pool
    const int64_t units = (int64_t)n_req * n_layers * n_heads;
    const int64_t entries = (int64_t)pool_size * n_layers * n_heads;
    const int nl = fam == HYPIC_DIAG ? d_k : 1;
    auto overlaps = [](const void *x, size_t xb, const void *y, size_t yb) {
        if (!x || !y) return false;
        const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(y);
        return a < b + yb && b < a + xb;
    };
    const size_t sb = (size_t)units * d_k * d_v * 4, mb = (size_t)units * d_k * d_k * 4, lb = (size_t)units * nl * 4;
    const size_t psb = (size_t)entries * d_k * d_v * 4, pmb = (size_t)entries * d_k * d_k * 4,
                 plb = (size_t)entries * nl * 4;
    const void *outs[] = {S_out, M_out, lam_out};
    const size_t outb[] = {sb, mb, lb};
    const void *ins[] = {pool_S, pool_M, pool_lam};
    const size_t inb[] = {psb, pmb, plb};
    for (int x = 0; x < 3; ++x) {
        for (int y = 0; y < 3; ++y)
            if (overlaps(outs[x], outb[x], ins[y], inb[y])) return HYPIC_EINVAL;
        for (int y = x + 1; y < 3; ++y)
            if (overlaps(outs[x], outb[x], outs[y], outb[y])) return HYPIC_EINVAL;
    }

    hypic::ChainArgs a;
    a.fam = compose_family(fam);
    a.R = n_req;
    a.n_layers = n_layers;
    a.H = n_heads;
    a.dk = d_k;
    a.dv = d_v;
    a.max_chain = max_chain;
    a.P = pool_size;
    a.chain_len = chain_len;
    a.seg_idx = seg_idx;
    a.pool_lam = pool_lam;
    a.pool_M = pool_M;
    a.pool_S = pool_S;
    a.S_init = nullptr;
    a.S_out = S_out;
    a.d_err = d_err;
    return from_cuda(hypic::launch_compose_prefix(a, lam_out, M_out, static_cast<cudaStream_t>(cuda_stream)));
}

}  // extern "C"
