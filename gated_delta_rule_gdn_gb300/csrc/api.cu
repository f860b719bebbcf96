// C ABI of libgdn_gb300.so (declared in include/gdn.h): argument checks, error reporting and
// kernel dispatch.  All buffers belong to the caller; the only allocation is the two-pass workspace when
// the caller passes none, made and freed on the call's stream.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/gdn.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;
thread_local int g_test_injection = 0;

gdn_status fail(gdn_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

gdn_status ok() {
    g_last_error.clear();
    return GDN_OK;
}

gdn_status cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dtype_ok(gdn_dtype d) { return d == GDN_F32 || d == GDN_BF16; }

gdn_status check_chunk(const gdn::ChunkArgs& a, gdn_dtype dtype, gdn_dtype o_dtype, int output_final_state,
                       const char* fn) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!dtype_ok(o_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown o_dtype %d", fn, (int)o_dtype);
    if (a.B < 1 || a.T < 0 || a.H < 1)
        return fail(GDN_ERR_INVALID_ARG, "%s: need B >= 1, T >= 0, H >= 1 (got B=%d T=%d H=%d)", fn, a.B, a.T, a.H);
    if (a.dk < 1 || a.dv < 1 || a.dk > 256 || a.dv > 256)
        return fail(GDN_ERR_UNSUPPORTED, "%s: head sizes must be 1..256 (got d_k=%d d_v=%d)", fn, a.dk, a.dv);
    if (a.C != 16 && a.C != 32 && a.C != 64)
        return fail(GDN_ERR_UNSUPPORTED, "%s: chunk_size must be 16, 32 or 64 (got %d)", fn, a.C);
    if (!std::isfinite(a.scale)) return fail(GDN_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if ((output_final_state != 0) != (a.hT != nullptr))
        return fail(GDN_ERR_INVALID_ARG, "%s: final_state must be non-NULL exactly when output_final_state is set", fn);
    if (a.cu) {
        if (a.B != 1) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens needs B == 1 (got B=%d)", fn, a.B);
        if (a.n_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens needs n_seqs >= 1 (got %d)", fn, a.n_seqs);
        if (!aligned(a.cu, 4)) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens is not 4-byte aligned", fn);
    }
    const bool any_tokens = (long)a.B * a.T > 0;
    if (any_tokens && (!a.q || !a.k || !a.v || !a.g || !a.beta || !a.o))
        return fail(GDN_ERR_INVALID_ARG, "%s: q, k, v, g, beta and o must be non-NULL", fn);
    const size_t es = dtype == GDN_BF16 ? 2 : 4;
    const size_t oes = o_dtype == GDN_BF16 ? 2 : 4;
    if (any_tokens && (!aligned(a.q, es) || !aligned(a.k, es) || !aligned(a.v, es) || !aligned(a.o, oes) ||
                       !aligned(a.g, 4) || !aligned(a.beta, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: a tensor is not aligned to its element size", fn);
    if ((a.h0 && !aligned(a.h0, 4)) || (a.hT && !aligned(a.hT, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: a state buffer is not 4-byte aligned", fn);
    if ((long)a.B * a.T * a.H > (1L << 31) / (a.dk > a.dv ? a.dk : a.dv))
        return fail(GDN_ERR_UNSUPPORTED, "%s: tensor has 2^31 elements or more", fn);
    return GDN_OK;
}

// Resolve a kernel request against what each kernel supports.  AUTO takes the two-pass tcgen05 path where it
// applies, else the generic one.  GDN_ALGO_TCGEN05 (the retired single-launch kernel) is refused.
gdn_status resolve_algo(const gdn::ChunkArgs& a, gdn_algo algo, const char* fn, gdn_algo* chosen) {
    if (algo != GDN_ALGO_AUTO && algo != GDN_ALGO_GENERIC && algo != GDN_ALGO_TCGEN05 && algo != GDN_ALGO_TWO_PASS)
        return fail(GDN_ERR_INVALID_ARG, "%s: unknown algo %d", fn, (int)algo);
    if (algo == GDN_ALGO_TCGEN05)
        return fail(GDN_ERR_UNSUPPORTED, "%s: the single-launch tcgen05 kernel was retired; use GDN_ALGO_TWO_PASS or "
                    "GDN_ALGO_AUTO", fn);
    const char* why_tp = gdn::two_pass_unsupported_reason(a);
    if (algo == GDN_ALGO_TWO_PASS && why_tp)
        return fail(GDN_ERR_UNSUPPORTED, "%s: the two-pass kernels do not apply: %s", fn, why_tp);
    if (algo == GDN_ALGO_AUTO) algo = !why_tp ? GDN_ALGO_TWO_PASS : GDN_ALGO_GENERIC;
    if (algo == GDN_ALGO_GENERIC) {
        const size_t need = gdn::generic_smem_bytes(a);
        if (need > gdn::kMaxSmemPerBlock)
            return fail(GDN_ERR_UNSUPPORTED,
                        "%s: the generic kernel would need %zu bytes of shared memory for d_k=%d, chunk_size=%d%s "
                        "(at most %zu); use a smaller chunk_size", fn, need, a.dk, a.C,
                        a.per_channel ? " and the per-channel gate" : "", gdn::kMaxSmemPerBlock);
    }
    *chosen = algo;
    return GDN_OK;
}

// Validate an optional activation descriptor and copy it into the kernel arguments.
gdn_status set_act(gdn::GateAct& dst, const gdn_gate_act* act, const char* fn) {
    dst = gdn::GateAct{nullptr, nullptr, 0};
    if (!act) return GDN_OK;
    if (act->dt_bias && !act->A_log)
        return fail(GDN_ERR_INVALID_ARG, "%s: dt_bias is given without A_log", fn);
    if ((act->A_log && !aligned(act->A_log, 4)) || (act->dt_bias && !aligned(act->dt_bias, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: A_log or dt_bias is not 4-byte aligned", fn);
    if (act->beta_sigmoid < 0 || act->beta_sigmoid > 2)
        return fail(GDN_ERR_INVALID_ARG, "%s: beta_sigmoid must be 0, 1 or 2 (got %d)", fn, act->beta_sigmoid);
    dst = gdn::GateAct{act->A_log, act->dt_bias, act->beta_sigmoid};
    return GDN_OK;
}

gdn_status chunk_common(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                        const float* initial_state, int output_final_state, float* final_state,
                        const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                        int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, gdn_algo algo, void* workspace,
                        size_t workspace_bytes, void* stream, bool per_channel, const char* fn,
                        const gdn_gate_act* act = nullptr, int H_k = 0) {
    gdn::ChunkArgs a{q, k, v, g, beta, scale, initial_state, final_state, cu_seqlens, n_seqs, o,
                     B, T, H, d_k, d_v, chunk_size, dtype == GDN_BF16 ? 1 : 0, per_channel ? 1 : 0,
                     o_dtype == GDN_F32 ? 1 : 0, gdn::GateAct{nullptr, nullptr, 0}, 0};
    gdn_status st = check_chunk(a, dtype, o_dtype, output_final_state, fn);
    if (st != GDN_OK) return st;
    if (H_k < 0 || (H_k > 0 && H % H_k != 0))
        return fail(GDN_ERR_INVALID_ARG, "%s: the value heads (%d) must be a multiple of the key heads (%d)", fn, H,
                    H_k);
    a.Hk = H_k;
    st = set_act(a.act, act, fn);
    if (st != GDN_OK) return st;
    gdn_algo chosen = GDN_ALGO_GENERIC;
    st = resolve_algo(a, algo, fn, &chosen);
    if (st != GDN_OK) return st;
    if (a.act.any() && chosen != GDN_ALGO_TWO_PASS)
        return fail(GDN_ERR_UNSUPPORTED, "%s: the gate and beta activation run on the two-pass path only (bf16, chunk 64, "
                    "d = 128, or d = 256 with the scalar gate)", fn);
    if (a.HK() != a.H && chosen != GDN_ALGO_TWO_PASS)
        return fail(GDN_ERR_UNSUPPORTED, "%s: grouped value heads run on the two-pass path only (bf16, chunk 64, d = 128, "
                    "or d = 256 with the scalar gate)", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (chosen == GDN_ALGO_TWO_PASS) {
        if (gdn::take_test_injection(GDN_TEST_FWD_RECORD_STALL)) a.test_fwd = 1;
        else if (!a.per_channel && gdn::take_test_injection(GDN_TEST_FWD_ONE_STAGE)) a.test_fwd = 2;
        const size_t need = gdn::two_pass_workspace_bytes(a);
        if (workspace && workspace_bytes < need)
            return fail(GDN_ERR_INVALID_ARG, "%s: workspace of %zu bytes is smaller than the %zu needed", fn,
                        workspace_bytes, need);
        if (workspace && !aligned(workspace, 256))
            return fail(GDN_ERR_INVALID_ARG, "%s: workspace is not 256-byte aligned", fn);
        void* ws = workspace;
        if (!ws && need > 0) {
            e = cudaMallocAsync(&ws, need, s);
            if (e != cudaSuccess) return cuda_fail(e, fn);
        }
        e = gdn::launch_chunk_two_pass(a, ws, ws ? (workspace ? workspace_bytes : need) : 0, s);
        if (!workspace && ws) {
            const cudaError_t e2 = cudaFreeAsync(ws, s);
            if (e == cudaSuccess) e = e2;
        }
    } else {
        e = gdn::launch_chunk_generic(a, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

// Stand-in arguments for the planning queries: pointers 256-byte aligned and never dereferenced.
gdn::ChunkArgs plan_args(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                         gdn_dtype o_dtype, int n_seqs) {
    const void* p = reinterpret_cast<const void*>(uintptr_t(1) << 20);
    float* fp = reinterpret_cast<float*>(uintptr_t(1) << 20);
    return gdn::ChunkArgs{p, p, p, fp, fp, 1.0f, nullptr, nullptr,
                          n_seqs > 0 ? reinterpret_cast<const int32_t*>(p) : nullptr, n_seqs > 0 ? n_seqs : 0,
                          const_cast<void*>(p), B, T, H, d_k, d_v, chunk_size, dtype == GDN_BF16 ? 1 : 0,
                          per_channel ? 1 : 0, o_dtype == GDN_F32 ? 1 : 0, gdn::GateAct{nullptr, nullptr, 0}, 0};
}

gdn_status step_common(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                       float* state, void* o, int N, int H, int d_k, int d_v, gdn_dtype dtype, gdn_dtype o_dtype,
                       void* stream, bool per_channel, const char* fn, const gdn_gate_act* act = nullptr,
                       int H_k = 0) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!dtype_ok(o_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown o_dtype %d", fn, (int)o_dtype);
    if (N < 1 || H < 1) return fail(GDN_ERR_INVALID_ARG, "%s: need N >= 1, H >= 1 (got N=%d H=%d)", fn, N, H);
    if (d_k < 1 || d_v < 1 || d_k > 256 || d_v > 256)
        return fail(GDN_ERR_UNSUPPORTED, "%s: head sizes must be 1..256 (got d_k=%d d_v=%d)", fn, d_k, d_v);
    if (!q || !k || !v || !g || !beta || !state || !o)
        return fail(GDN_ERR_INVALID_ARG, "%s: q, k, v, g, beta, state and o must be non-NULL", fn);
    if (!std::isfinite(scale)) return fail(GDN_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    const size_t es = dtype == GDN_BF16 ? 2 : 4;
    const size_t oes = o_dtype == GDN_BF16 ? 2 : 4;
    if (!aligned(q, es) || !aligned(k, es) || !aligned(v, es) || !aligned(o, oes) || !aligned(g, 4) ||
        !aligned(beta, 4) || !aligned(state, 4))
        return fail(GDN_ERR_INVALID_ARG, "%s: a tensor is not aligned to its element size", fn);
    if ((long)N * H > (1L << 31) / ((long)d_k * d_v))
        return fail(GDN_ERR_UNSUPPORTED, "%s: state has 2^31 elements or more", fn);
    gdn::StepArgs a{q, k, v, g, beta, scale, state, o, N, H, d_k, d_v, dtype == GDN_BF16 ? 1 : 0,
                    o_dtype == GDN_F32 ? 1 : 0, per_channel ? 1 : 0, gdn::GateAct{nullptr, nullptr, 0}, 0};
    gdn_status st = set_act(a.act, act, fn);
    if (st != GDN_OK) return st;
    if (per_channel && a.act.gate())
        return fail(GDN_ERR_UNSUPPORTED, "%s: the gate activation applies to the scalar gate only", fn);
    if (H_k < 0 || (H_k > 0 && H % H_k != 0))
        return fail(GDN_ERR_INVALID_ARG, "%s: the value heads (%d) must be a multiple of the key heads (%d)", fn, H,
                    H_k);
    a.Hk = H_k;
    cudaError_t e = gdn::launch_recurrent_step(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}


// Validate a backward request (everything except the pointers' contents) and settle its chunk.
gdn_status check_bwd(gdn::BwdArgs& a, gdn_dtype dtype, gdn_dtype do_dtype, const char* fn) {
    if (!dtype_ok(dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!dtype_ok(do_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: unknown do_dtype %d", fn, (int)do_dtype);
    if (a.B < 1 || a.T < 0 || a.H < 1)
        return fail(GDN_ERR_INVALID_ARG, "%s: need B >= 1, T >= 0, H >= 1 (got B=%d T=%d H=%d)", fn, a.B, a.T, a.H);
    if (a.dk < 1 || a.dv < 1 || a.dk > 256 || a.dv > 256)
        return fail(GDN_ERR_UNSUPPORTED, "%s: head sizes must be 1..256 (got d_k=%d d_v=%d)", fn, a.dk, a.dv);
    if (a.C == 0) {
        a.C = gdn::bwd_auto_chunk(a.dk, a.per_channel != 0);
        if (a.C == 0)
            return fail(GDN_ERR_UNSUPPORTED, "%s: no chunk_size fits the shared memory of one CTA for d_k=%d", fn,
                        a.dk);
    }
    if (a.C != 16 && a.C != 32)
        return fail(GDN_ERR_UNSUPPORTED, "%s: chunk_size must be 16, 32 or 0 (got %d)", fn, a.C);
    const size_t need = gdn::bwd_smem_bytes(a.C, a.dk, a.per_channel != 0);
    if (need > gdn::kMaxSmemPerBlock)
        return fail(GDN_ERR_UNSUPPORTED,
                    "%s: the backward would need %zu bytes of shared memory for d_k=%d, chunk_size=%d (at most %zu); "
                    "use a smaller chunk_size", fn, need, a.dk, a.C, gdn::kMaxSmemPerBlock);
    if (!std::isfinite(a.scale)) return fail(GDN_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (a.cu) {
        if (a.B != 1) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens needs B == 1 (got B=%d)", fn, a.B);
        if (a.n_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens needs n_seqs >= 1 (got %d)", fn, a.n_seqs);
        if (!aligned(a.cu, 4)) return fail(GDN_ERR_INVALID_ARG, "%s: cu_seqlens is not 4-byte aligned", fn);
    }
    if ((long)a.B * a.T * a.H > (1L << 31) / (a.dk > a.dv ? a.dk : a.dv))
        return fail(GDN_ERR_UNSUPPORTED, "%s: tensor has 2^31 elements or more", fn);
    return GDN_OK;
}

}  // namespace

namespace gdn {
bool take_test_injection(int what) {
    if (g_test_injection != what) return false;
    g_test_injection = 0;
    return true;
}
}  // namespace gdn

extern "C" {

gdn_status gdn_chunk_fwd_algo(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, const float* initial_state, int output_final_state,
                              float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T,
                              int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                              gdn_algo algo, void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, algo, nullptr, 0, stream, false,
                        "gdn_chunk_fwd");
}

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                         const float* initial_state, int output_final_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                         int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, void* stream) {
    return gdn_chunk_fwd_algo(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens,
                              n_seqs, o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, GDN_ALGO_AUTO, stream);
}

gdn_status kda_chunk_fwd_algo(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, const float* initial_state, int output_final_state,
                              float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T,
                              int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                              gdn_algo algo, void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, algo, nullptr, 0, stream, true,
                        "kda_chunk_fwd");
}

gdn_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                         const float* initial_state, int output_final_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                         int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, void* stream) {
    return kda_chunk_fwd_algo(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens,
                              n_seqs, o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, GDN_ALGO_AUTO, stream);
}

gdn_status gdn_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            float scale, const float* initial_state, int output_final_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                            int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, gdn_algo algo, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, algo, workspace, workspace_bytes, stream,
                        false, "gdn_chunk_fwd");
}

gdn_status kda_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            float scale, const float* initial_state, int output_final_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                            int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, gdn_algo algo, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, algo, workspace, workspace_bytes, stream,
                        true, "kda_chunk_fwd");
}

gdn_status gdn_chunk_fwd_noalloc(int per_channel, const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float scale, const float* initial_state, int output_final_state,
                                 float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T,
                                 int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                                 void* stream) {
    const char* fn = "gdn_chunk_fwd_noalloc";
    gdn::ChunkArgs a{q, k, v, g, beta, scale, initial_state, final_state, cu_seqlens, n_seqs, o,
                     B, T, H, d_k, d_v, chunk_size, dtype == GDN_BF16 ? 1 : 0, per_channel ? 1 : 0,
                     o_dtype == GDN_F32 ? 1 : 0, gdn::GateAct{nullptr, nullptr, 0}, 0};
    gdn_status st = check_chunk(a, dtype, o_dtype, output_final_state, fn);
    if (st != GDN_OK) return st;
    if (const char* why = gdn::two_pass_unsupported_reason(a))
        return fail(GDN_ERR_UNSUPPORTED, "%s: the two-pass kernels do not apply: %s", fn, why);
    const size_t need = gdn::two_pass_workspace_bytes(a), cap = gdn::static_workspace_capacity();
    if (need > cap)
        return fail(GDN_ERR_UNSUPPORTED,
                    "%s: the request needs %zu bytes of scratch; the static scratch holds %zu (use gdn_chunk_fwd_ws "
                    "with a caller workspace)", fn, need, cap);
    void* ws = nullptr;
    cudaError_t e = gdn::static_workspace(&ws);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    e = gdn::launch_chunk_two_pass(a, ws, cap, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

gdn_status gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, float* state, void* o, int N, int H, int d_k, int d_v, gdn_dtype dtype,
                              gdn_dtype o_dtype, void* stream) {
    return step_common(q, k, v, g, beta, scale, state, o, N, H, d_k, d_v, dtype, o_dtype, stream, false,
                       "gdn_recurrent_step");
}

gdn_status gdn_chunk_fwd_act(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             float scale, const float* initial_state, int output_final_state, float* final_state,
                             const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H, int d_k, int d_v,
                             int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype, const gdn_gate_act* act,
                             gdn_algo algo, void* workspace, size_t workspace_bytes, void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, algo, workspace, workspace_bytes, stream,
                        false, "gdn_chunk_fwd_act", act);
}

gdn_status gdn_chunk_fwd_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, const float* initial_state, int output_final_state,
                            float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o, int B, int T, int H_k,
                            int H_v, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                            const gdn_gate_act* act, gdn_algo algo, void* workspace, size_t workspace_bytes,
                            void* stream) {
    return chunk_common(q, k, v, g, beta, scale, initial_state, output_final_state, final_state, cu_seqlens, n_seqs,
                        o, B, T, H_v, d_k, d_v, chunk_size, dtype, o_dtype, algo, workspace, workspace_bytes, stream,
                        per_channel != 0, "gdn_chunk_fwd_ex", act, H_k);
}

gdn_status gdn_recurrent_step_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float scale, float* state, void* o, int N, int H_k, int H_v,
                                 int d_k, int d_v, gdn_dtype dtype, gdn_dtype o_dtype, const gdn_gate_act* act,
                                 void* stream) {
    return step_common(q, k, v, g, beta, scale, state, o, N, H_v, d_k, d_v, dtype, o_dtype, stream, per_channel != 0,
                       "gdn_recurrent_step_ex", act, H_k);
}

gdn_status gdn_recurrent_step_act(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  float scale, float* state, void* o, int N, int H, int d_k, int d_v,
                                  gdn_dtype dtype, gdn_dtype o_dtype, const gdn_gate_act* act, void* stream) {
    return step_common(q, k, v, g, beta, scale, state, o, N, H, d_k, d_v, dtype, o_dtype, stream, false,
                       "gdn_recurrent_step_act", act);
}

gdn_status kda_recurrent_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, float* state, void* o, int N, int H, int d_k, int d_v, gdn_dtype dtype,
                              gdn_dtype o_dtype, void* stream) {
    return step_common(q, k, v, g, beta, scale, state, o, N, H, d_k, d_v, dtype, o_dtype, stream, true,
                       "kda_recurrent_step");
}

gdn_status gdn_chunk_plan(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                          gdn_dtype o_dtype, int varlen, gdn_algo requested, gdn_algo* chosen) {
    const char* fn = "gdn_chunk_plan";
    if (!chosen) return fail(GDN_ERR_INVALID_ARG, "%s: chosen is NULL", fn);
    const gdn::ChunkArgs a = plan_args(per_channel, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, varlen ? 1 : 0);
    gdn_status st = check_chunk(a, dtype, o_dtype, 0, fn);
    if (st != GDN_OK) return st;
    gdn_algo c = GDN_ALGO_GENERIC;
    st = resolve_algo(a, requested, fn, &c);
    if (st != GDN_OK) return st;
    *chosen = c;
    return ok();
}

gdn_status gdn_chunk_workspace_size(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size,
                                    gdn_dtype dtype, gdn_dtype o_dtype, int n_seqs, gdn_algo requested,
                                    size_t* bytes) {
    const char* fn = "gdn_chunk_workspace_size";
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, "%s: bytes is NULL", fn);
    if (n_seqs < 0) return fail(GDN_ERR_INVALID_ARG, "%s: n_seqs must be >= 0 (got %d)", fn, n_seqs);
    const gdn::ChunkArgs a = plan_args(per_channel, B, T, H, d_k, d_v, chunk_size, dtype, o_dtype, n_seqs);
    gdn_status st = check_chunk(a, dtype, o_dtype, 0, fn);
    if (st != GDN_OK) return st;
    gdn_algo c = GDN_ALGO_GENERIC;
    st = resolve_algo(a, requested, fn, &c);
    if (st != GDN_OK) return st;
    *bytes = c == GDN_ALGO_TWO_PASS ? gdn::two_pass_workspace_bytes(a) : 0;
    return ok();
}

gdn_status gdn_chunk_bwd_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, const float* initial_state, const void* grad_o,
                            const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                            float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                            float* grad_A_log, float* grad_dt_bias, int B, int T, int H_k, int H, int d_k, int d_v,
                            int chunk_size, gdn_dtype dtype, gdn_dtype do_dtype, const gdn_gate_act* act,
                            void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "gdn_chunk_bwd";
    gdn::BwdArgs a{q, k, v, g, beta, scale, initial_state, grad_o, grad_final_state, cu_seqlens, n_seqs,
                   grad_q, grad_k, grad_v, grad_g, grad_beta, grad_initial_state, nullptr,
                   B, T, H, d_k, d_v, chunk_size, dtype == GDN_BF16 ? 1 : 0, do_dtype == GDN_BF16 ? 1 : 0,
                   per_channel ? 1 : 0, 0, 0, nullptr, nullptr};
    gdn_status st = check_bwd(a, dtype, do_dtype, fn);
    if (st != GDN_OK) return st;
    if (H_k < 0 || (H_k > 0 && H % H_k != 0))
        return fail(GDN_ERR_INVALID_ARG, "%s: the value heads (%d) must be a multiple of the key heads (%d)", fn, H,
                    H_k);
    a.Hk = H_k;
    gdn::GateAct ga{nullptr, nullptr, 0};
    st = set_act(ga, act, fn);
    if (st != GDN_OK) return st;
    if (per_channel && ga.gate())
        return fail(GDN_ERR_UNSUPPORTED, "%s: the gate activation applies to the scalar gate only", fn);
    if (ga.gate() && (!grad_A_log || !aligned(grad_A_log, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: grad_A_log must be a 4-byte aligned [H] buffer when A_log is given", fn);
    if (grad_dt_bias && (!ga.dt_bias || !aligned(grad_dt_bias, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: grad_dt_bias needs dt_bias and 4-byte alignment", fn);
    const bool any_tokens = (long)a.B * a.T > 0;
    if (any_tokens && (!q || !k || !v || !g || !beta || !grad_o || !grad_q || !grad_k || !grad_v || !grad_g ||
                       !grad_beta))
        return fail(GDN_ERR_INVALID_ARG, "%s: q, k, v, g, beta, grad_o and the token gradients must be non-NULL", fn);
    const size_t es = dtype == GDN_BF16 ? 2 : 4, des = do_dtype == GDN_BF16 ? 2 : 4;
    if (any_tokens && (!aligned(q, es) || !aligned(k, es) || !aligned(v, es) || !aligned(grad_o, des) ||
                       !aligned(g, 4) || !aligned(beta, 4) || !aligned(grad_q, 4) || !aligned(grad_k, 4) ||
                       !aligned(grad_v, 4) || !aligned(grad_g, 4) || !aligned(grad_beta, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: a tensor is not aligned to its element size", fn);
    if ((initial_state && !aligned(initial_state, 4)) || (grad_final_state && !aligned(grad_final_state, 4)) ||
        (grad_initial_state && !aligned(grad_initial_state, 4)))
        return fail(GDN_ERR_INVALID_ARG, "%s: a state buffer is not 4-byte aligned", fn);
    const size_t need = gdn::bwd_workspace_bytes(a);
    if (workspace && workspace_bytes < need)
        return fail(GDN_ERR_INVALID_ARG, "%s: workspace of %zu bytes is smaller than the %zu needed", fn,
                    workspace_bytes, need);
    if (workspace && !aligned(workspace, 256))
        return fail(GDN_ERR_INVALID_ARG, "%s: workspace is not 256-byte aligned", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    cudaError_t e = cudaSuccess;
    if (!ws && need > 0) {
        e = cudaMallocAsync(&ws, need, s);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    a.ck = static_cast<float*>(ws);
    a.test_skip_record = gdn::take_test_injection(GDN_TEST_BWD_RECORD_STALL) ? 1 : 0;
    if (a.HK() < a.H) {
        a.gq_part = reinterpret_cast<float*>(static_cast<char*>(ws) + gdn::bwd_part_offset(a));
        a.gk_part = a.gq_part + (size_t)a.B * a.T * a.H * a.dk;
    }
    const long n_tok = (long)a.B * a.T * a.H;
    float* g_act = reinterpret_cast<float*>(static_cast<char*>(ws) + gdn::bwd_act_offset(a));
    float* beta_act = g_act + n_tok;
    if (ga.any()) {
        e = gdn::launch_bwd_act_apply(g, beta, ga, g_act, beta_act, n_tok, H, s);
        if (ga.gate()) a.g = g_act;
        if (ga.beta_sigmoid) a.beta = beta_act;
    }
    if (e == cudaSuccess) e = gdn::launch_chunk_bwd(a, s);
    if (e == cudaSuccess) e = gdn::launch_bwd_group_sum(a, s);
    if (e == cudaSuccess && ga.any())
        e = gdn::launch_bwd_act_post(g, beta, g_act, ga, grad_g, grad_beta, grad_A_log, grad_dt_bias,
                                     (long)a.B * a.T, H, s);
    if (!workspace && ws) {
        const cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

gdn_status gdn_chunk_bwd_act(int per_channel, const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float scale, const float* initial_state, const void* grad_o,
                             const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                             float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                             float* grad_A_log, float* grad_dt_bias, int B, int T, int H, int d_k, int d_v,
                             int chunk_size, gdn_dtype dtype, gdn_dtype do_dtype, const gdn_gate_act* act,
                             void* workspace, size_t workspace_bytes, void* stream) {
    return gdn_chunk_bwd_ex(per_channel, q, k, v, g, beta, scale, initial_state, grad_o, grad_final_state,
                            cu_seqlens, n_seqs, grad_q, grad_k, grad_v, grad_g, grad_beta, grad_initial_state,
                            grad_A_log, grad_dt_bias, B, T, 0, H, d_k, d_v, chunk_size, dtype, do_dtype, act,
                            workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_bwd(int per_channel, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, float scale, const float* initial_state, const void* grad_o,
                         const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                         float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                         int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                         gdn_dtype do_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    return gdn_chunk_bwd_ex(per_channel, q, k, v, g, beta, scale, initial_state, grad_o, grad_final_state,
                            cu_seqlens, n_seqs, grad_q, grad_k, grad_v, grad_g, grad_beta, grad_initial_state,
                            nullptr, nullptr, B, T, 0, H, d_k, d_v, chunk_size, dtype, do_dtype, nullptr, workspace,
                            workspace_bytes, stream);
}

gdn_status gdn_chunk_bwd_workspace_size_ex(int per_channel, int B, int T, int H_k, int H, int d_k, int d_v,
                                           int chunk_size, int n_seqs, size_t* bytes) {
    const char* fn = "gdn_chunk_bwd_workspace_size";
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, "%s: bytes is NULL", fn);
    if (n_seqs < 0) return fail(GDN_ERR_INVALID_ARG, "%s: n_seqs must be >= 0 (got %d)", fn, n_seqs);
    const int32_t* cu = n_seqs > 0 ? reinterpret_cast<const int32_t*>(uintptr_t(1) << 20) : nullptr;
    gdn::BwdArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, 1.0f, nullptr, nullptr, nullptr, cu, n_seqs,
                   nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                   B, T, H, d_k, d_v, chunk_size, 0, 0, per_channel ? 1 : 0, 0, 0, nullptr, nullptr};
    gdn_status st = check_bwd(a, GDN_F32, GDN_F32, fn);
    if (st != GDN_OK) return st;
    if (H_k < 0 || (H_k > 0 && H % H_k != 0))
        return fail(GDN_ERR_INVALID_ARG, "%s: the value heads (%d) must be a multiple of the key heads (%d)", fn, H,
                    H_k);
    a.Hk = H_k;
    *bytes = gdn::bwd_workspace_bytes(a);
    return ok();
}

gdn_status gdn_chunk_bwd_workspace_size(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size,
                                        int n_seqs, size_t* bytes) {
    return gdn_chunk_bwd_workspace_size_ex(per_channel, B, T, 0, H, d_k, d_v, chunk_size, n_seqs, bytes);
}

gdn_status gdn_test_inject(int what) {
    if (what != 0 && what != GDN_TEST_BWD_RECORD_STALL && what != GDN_TEST_FWD_RECORD_STALL &&
        what != GDN_TEST_FWD_ONE_STAGE)
        return fail(GDN_ERR_INVALID_ARG, "gdn_test_inject: unknown injection %d", what);
    g_test_injection = what;
    return ok();
}

const char* gdn_last_error(void) { return g_last_error.c_str(); }

gdn_status gdn_device_status(int clear) {
    unsigned tp = 0, gt = 0, bw = 0, d2 = 0;
    cudaError_t e = gdn::tp_read_and_clear_status(&tp, clear != 0);
    if (e == cudaSuccess) e = gdn::gt_read_and_clear_status(&gt, clear != 0);
    if (e == cudaSuccess) e = gdn::d256_read_and_clear_status(&d2, clear != 0);
    gt |= d2;   // the scalar-gate forward at either head size
    if (e == cudaSuccess) e = gdn::bwd_read_and_clear_status(&bw, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_device_status");
    const unsigned nf = gdn::kStatusNonfinite;
    if (((tp | gt) & ~nf) != 0 || bw != 0)
        return fail(GDN_ERR_TIMEOUT,
                    "gdn_device_status: a kernel gave up a bounded wait (per-channel forward 0x%x, scalar-gate forward "
                    "0x%x, backward 0x%x)", tp, gt, bw);
    if (((tp | gt) & nf) != 0)
        return fail(GDN_ERR_NONFINITE,
                    "gdn_device_status: a chunk forward wrote a non-finite value to o or the final state (an fp16 "
                    "operand passed 65504, or an input was not finite)");
    return ok();
}

const char* gdn_version(void) { return "gdn_gb300 0.1 (sm_103a)"; }

}  // extern "C"
