// api.cu -- the C ABI of libdspark.so (declared in include/dspark.h):
// argument validation, workspace carving, per-device launch configuration.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "dspark_internal.cuh"
#include "sts_fit.cuh"

namespace {

thread_local char g_err[512] = "";

// Bound of every device wait, read at each launch (dspark_set_wait_timeout_ns).
std::atomic<uint64_t> g_wait_ns{dspark::kWaitTimeoutNs};

dspark_status fail(dspark_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

dspark_status cuda_fail(cudaError_t e, const char *what) {
    return fail(DSPARK_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

size_t dtype_size(int32_t dt) { return dt == DSPARK_BF16 ? 2 : 4; }

// Per-device facts and one-time kernel attributes.
struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int verify_blocks[2] = {0, 0};  // per logit dtype (0 = fp32, 1 = bf16)
    int tail_blocks[2] = {0, 0};    // the small verify's tail kernel, per logit dtype
    int score_blocks[2] = {0, 0};   // per hidden dtype
    int entropy_blocks[2] = {0, 0}; // per logit dtype
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

dspark_status device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(DSPARK_EDEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return fail(DSPARK_EDEVICE, "libdspark is built for sm_103a; device %d is sm_%d%d", dev,
                        major, minor);
        for (int bf = 0; bf < 2; ++bf) {
            d.verify_blocks[bf] = dspark::verify_blocks_per_sm(bf);
            if (d.verify_blocks[bf] <= 0)
                return fail(DSPARK_ECUDA, "verify kernel cannot be resident (smem %zu bytes)",
                            dspark::verify_smem_bytes());
            d.tail_blocks[bf] = dspark::verify_tail_blocks_per_sm(bf);
            if (d.tail_blocks[bf] <= 0)
                return fail(DSPARK_ECUDA, "verify tail kernel cannot be resident");
            d.score_blocks[bf] = dspark::score_blocks_per_sm(bf);
            if (d.score_blocks[bf] <= 0)
                return fail(DSPARK_ECUDA, "score kernel cannot be resident");
            d.entropy_blocks[bf] = dspark::entropy_blocks_per_sm(bf);
            if (d.entropy_blocks[bf] <= 0)
                return fail(DSPARK_ECUDA, "entropy score kernel cannot be resident");
        }
        d.ready = true;
    }
    *out = &d;
    return DSPARK_OK;
}

dspark_status check_shape(const dspark_step *s) {
    if (!s) return fail(DSPARK_EINVAL, "step is NULL");
    if (s->B < 0 || s->B > DSPARK_MAX_B) return fail(DSPARK_EINVAL, "B=%d outside [0, %d]", s->B, DSPARK_MAX_B);
    if (s->gamma < 1 || s->gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_EINVAL, "gamma=%d outside [1, %d]", s->gamma, DSPARK_MAX_GAMMA);
    if (s->V < 1 || s->V > DSPARK_MAX_V) return fail(DSPARK_EINVAL, "V=%d outside [1, %d]", s->V, DSPARK_MAX_V);
    if (s->d < 1 || s->d > DSPARK_MAX_D) return fail(DSPARK_EINVAL, "d=%d outside [1, %d]", s->d, DSPARK_MAX_D);
    if (s->logit_dtype != DSPARK_F32 && s->logit_dtype != DSPARK_BF16)
        return fail(DSPARK_EDTYPE, "logit_dtype=%d", s->logit_dtype);
    if (s->hidden_dtype != DSPARK_F32 && s->hidden_dtype != DSPARK_BF16)
        return fail(DSPARK_EDTYPE, "hidden_dtype=%d", s->hidden_dtype);
    return DSPARK_OK;
}

dspark_status check_workspace(const dspark_step *s, dspark::WorkspaceLayout *lay) {
    *lay = dspark::workspace_layout(s->B, s->gamma, s->V);
    if (!s->workspace) return fail(DSPARK_EWORKSPACE, "workspace is NULL");
    if (!aligned(s->workspace, 256)) return fail(DSPARK_EWORKSPACE, "workspace is not 256-byte aligned");
    if (s->workspace_bytes < lay->total)
        return fail(DSPARK_EWORKSPACE, "workspace has %zu bytes, needs %zu", s->workspace_bytes, lay->total);
    return DSPARK_OK;
}

template <typename T>
T *ws_at(const dspark_step *s, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(s->workspace) + off);
}

// One NVTX range per ABI call, named after the call: profilers (nsys, ncu's
// NVTX filters) see the step's structure.  Without a tool attached the
// push / pop are no-ops.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

#define REQUIRE(ptr)                                                             \
    do {                                                                         \
        if (!(ptr)) return fail(DSPARK_EINVAL, "%s: " #ptr " is NULL", fn);     \
    } while (0)
#define REQUIRE_ALIGNED(ptr, n)                                                  \
    do {                                                                         \
        if (!aligned((ptr), (n)))                                                \
            return fail(DSPARK_EALIGN, "%s: " #ptr " is not %d-byte aligned", fn, int(n)); \
    } while (0)

}  // namespace

extern "C" {

size_t dspark_workspace_size(int32_t B, int32_t gamma, int32_t V, int32_t d) {
    if (B < 0 || B > DSPARK_MAX_B || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 ||
        V > DSPARK_MAX_V || d < 1 || d > DSPARK_MAX_D)
        return 0;
    return dspark::workspace_layout(B, gamma, V).total;
}

dspark_status dspark_workspace_init(void *workspace, size_t workspace_bytes, dspark_stream_t stream) {
    if (!workspace) return fail(DSPARK_EWORKSPACE, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
    g_err[0] = 0;
    return DSPARK_OK;
}

// Steps a1-a3 (and, with pack, a4) of dspark_score_budget and
// dspark_score_compact.
static dspark_status score_impl(const dspark_step *s, bool pack, dspark_stream_t stream,
                                const char *fn) {
    dspark_status st = check_shape(s);
    if (st) return st;
    if (s->B == 0) return DSPARK_OK;
    REQUIRE(s->L);
    REQUIRE(s->draft_off);
    REQUIRE(s->row_off);
    if (pack) {
        REQUIRE(s->draft_tokens);
        REQUIRE(s->packed_ids);
        REQUIRE(s->packed_pos);
        REQUIRE(s->row_req);
        REQUIRE(s->row_k);
    }
    const bool fixed = s->fixed_budget >= 0;
    if (fixed && s->cap_T >= 0)
        return fail(DSPARK_EINVAL, "%s: a fixed budget (%d) cannot be combined with a cap (%d)", fn,
                    s->fixed_budget, s->cap_T);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    DeviceInfo *dev;
    if (fixed) {
        if ((st = device_info(&dev))) return st;
        dspark::FixedArgs a{s->B, s->gamma, s->fixed_budget, s->L, s->draft_off, s->row_off,
                            pack ? 1 : 0, s->draft_tokens, s->last_tokens, s->seq_lens_in,
                            s->packed_ids, s->packed_pos, s->row_req, s->row_k};
        cudaError_t e = dspark::launch_fixed_budget(a, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, pack ? "fixed_pack_kernel launch" : "fixed_budget_kernel launch");
        return DSPARK_OK;
    }
    REQUIRE(s->hidden);
    REQUIRE(s->head_w);
    REQUIRE(s->head_bias);
    REQUIRE(s->sts_tau);
    REQUIRE(s->conf);
    REQUIRE(s->survival);
    REQUIRE(s->L0);
    if (std::isnan(s->cost_c)) return fail(DSPARK_EINVAL, "%s: cost_c is NaN", fn);
    const size_t hs = dtype_size(s->hidden_dtype);
    REQUIRE_ALIGNED(s->hidden, 16);
    REQUIRE_ALIGNED(s->head_w, 16);
    if ((size_t(s->d) * hs) % 16 != 0)
        return fail(DSPARK_EALIGN, "%s: a hidden row (d=%d) is not a multiple of 16 bytes", fn, s->d);
    dspark::WorkspaceLayout lay;
    if ((st = check_workspace(s, &lay))) return st;
    if ((st = device_info(&dev))) return st;

    // One CTA per resident slot, each a contiguous range of the B*gamma rows.
    const long long rows = (long long)s->B * s->gamma;
    const int hb = s->hidden_dtype == DSPARK_BF16;
    const int grid = int(std::min<long long>(rows, (long long)dev->sms * dev->score_blocks[hb]));
    dspark::ScoreArgs a{};
    a.B = s->B; a.gamma = s->gamma; a.d = s->d;
    a.hidden_bf16 = s->hidden_dtype == DSPARK_BF16;
    a.hidden = s->hidden; a.head_w = s->head_w; a.head_bias = s->head_bias; a.sts_tau = s->sts_tau;
    a.cost_c = s->cost_c; a.cap_T = s->cap_T;
    a.conf = s->conf; a.survival = s->survival; a.L0 = s->L0; a.L = s->L;
    a.draft_off = s->draft_off; a.row_off = s->row_off;
    a.done_cnt = ws_at<int32_t>(s, lay.score_done);
    a.row_ctr = ws_at<int32_t>(s, lay.score_rows);
    a.status = ws_at<int32_t>(s, lay.status);
    a.wait_ns = g_wait_ns.load();
    if (pack) {
        a.pack = 1;
        a.draft_tokens = s->draft_tokens;
        a.last_tokens = s->last_tokens;
        a.seq_lens = s->seq_lens_in;
        a.packed_ids = s->packed_ids;
        a.packed_pos = s->packed_pos;
        a.row_req = s->row_req;
        a.row_k = s->row_k;
    }
    cudaError_t e = dspark::launch_score_budget(a, grid, cs);
    if (e != cudaSuccess) return cuda_fail(e, "score_budget_kernel launch");
    return DSPARK_OK;
}

dspark_status dspark_score_budget(const dspark_step *s, dspark_stream_t stream) {
    NvtxRange range("dspark_score_budget");
    return score_impl(s, false, stream, "dspark_score_budget");
}

dspark_status dspark_score_compact(const dspark_step *s, dspark_stream_t stream) {
    NvtxRange range("dspark_score_compact");
    return score_impl(s, true, stream, "dspark_score_compact");
}

dspark_status dspark_score_entropy(const dspark_step *s, float theta, dspark_stream_t stream) {
    NvtxRange range("dspark_score_entropy");
    const char *fn = "dspark_score_entropy";
    dspark_status st = check_shape(s);
    if (st) return st;
    if (!(theta > 0.0f) || std::isinf(theta))
        return fail(DSPARK_EINVAL, "%s: theta must be finite and > 0", fn);
    if (s->fixed_budget >= 0)
        return fail(DSPARK_EINVAL, "%s: a fixed budget has no confidences (use dspark_score_budget)",
                    fn);
    if (std::isnan(s->cost_c)) return fail(DSPARK_EINVAL, "%s: cost_c is NaN", fn);
    if (s->B == 0) return DSPARK_OK;
    REQUIRE(s->draft_logits);
    REQUIRE(s->conf);
    REQUIRE(s->survival);
    REQUIRE(s->L0);
    REQUIRE(s->L);
    REQUIRE(s->draft_off);
    REQUIRE(s->row_off);
    const size_t ls = dtype_size(s->logit_dtype);
    REQUIRE_ALIGNED(s->draft_logits, 16);
    if ((size_t(s->V) * ls) % 16 != 0)
        return fail(DSPARK_EALIGN, "%s: a logit row (V=%d) is not a multiple of 16 bytes", fn, s->V);
    dspark::WorkspaceLayout lay;
    if ((st = check_workspace(s, &lay))) return st;
    DeviceInfo *dev;
    if ((st = device_info(&dev))) return st;

    const long long rows = (long long)s->B * s->gamma;
    const int bf = s->logit_dtype == DSPARK_BF16;
    const int grid = int(std::min<long long>(rows, (long long)dev->sms * dev->entropy_blocks[bf]));
    dspark::ScoreArgs a{};
    a.B = s->B; a.gamma = s->gamma; a.d = s->V;
    a.hidden_bf16 = bf;
    a.hidden = s->draft_logits;
    a.ent_scale = float(1.4426950408889634 / double(theta));
    a.cost_c = s->cost_c; a.cap_T = s->cap_T;
    a.conf = s->conf; a.survival = s->survival; a.L0 = s->L0; a.L = s->L;
    a.draft_off = s->draft_off; a.row_off = s->row_off;
    a.done_cnt = ws_at<int32_t>(s, lay.score_done);
    a.row_ctr = ws_at<int32_t>(s, lay.score_rows);
    a.status = ws_at<int32_t>(s, lay.status);
    a.wait_ns = g_wait_ns.load();
    cudaError_t e = dspark::launch_score_entropy(a, grid, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "score_entropy_kernel launch");
    return DSPARK_OK;
}

dspark_status dspark_fit_sts_tau(int32_t N, int32_t gamma, const float *conf,
                                 const float *tau_used, const int32_t *L,
                                 const int32_t *accept_len, float tau_min, float tau_max,
                                 float *tau_out, float *nll_out, int32_t *n_obs,
                                 dspark_stream_t stream) {
    NvtxRange range("dspark_fit_sts_tau");
    const char *fn = "dspark_fit_sts_tau";
    if (N < 0) return fail(DSPARK_EINVAL, "%s: N=%d < 0", fn, N);
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_EINVAL, "%s: gamma=%d outside [1, %d]", fn, gamma, DSPARK_MAX_GAMMA);
    if (!(tau_min > 0.0f) || !(tau_max >= tau_min) || std::isinf(tau_max))
        return fail(DSPARK_EINVAL, "%s: need 0 < tau_min <= tau_max < inf", fn);
    REQUIRE(tau_used);
    REQUIRE(tau_out);
    if (N > 0) {
        REQUIRE(conf);
        REQUIRE(L);
        REQUIRE(accept_len);
    }
    DeviceInfo *dev;
    dspark_status st;
    if ((st = device_info(&dev))) return st;
    dspark::FitArgs a{N, gamma, conf, tau_used, L, accept_len, tau_min, tau_max,
                      tau_out, nll_out, n_obs};
    cudaError_t e = dspark::launch_sts_fit(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sts_fit_kernel launch");
    return DSPARK_OK;
}

dspark_status dspark_compact(const dspark_step *s, dspark_stream_t stream) {
    NvtxRange range("dspark_compact");
    const char *fn = "dspark_compact";
    dspark_status st = check_shape(s);
    if (st) return st;
    if (s->B == 0) return DSPARK_OK;
    REQUIRE(s->L);
    REQUIRE(s->row_off);
    REQUIRE(s->draft_tokens);
    REQUIRE(s->packed_ids);
    REQUIRE(s->packed_pos);
    REQUIRE(s->row_req);
    REQUIRE(s->row_k);
    DeviceInfo *dev;
    if ((st = device_info(&dev))) return st;
    dspark::CompactArgs a{s->B, s->gamma, s->L, s->row_off, s->draft_tokens, s->last_tokens,
                          s->seq_lens_in, s->packed_ids, s->packed_pos, s->row_req, s->row_k};
    cudaError_t e = dspark::launch_compact(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "compact_kernel launch");
    return DSPARK_OK;
}

}  // extern "C"

// The verify launch shared by dspark_verify (audit pointers NULL) and
// dspark_verify_cap_accept.
static dspark_status verify_impl(const dspark_step *s, const int32_t *commit_len,
                                 int32_t *accept_full, int32_t *audit_totals,
                                 dspark_stream_t stream, const char *fn) {
    dspark_status st = check_shape(s);
    if (st) return st;
    if (s->B == 0) return DSPARK_OK;
    const bool greedy = s->temperature == 0.0f;
    if (!(s->temperature >= 0.0f) || std::isinf(s->temperature))
        return fail(DSPARK_EINVAL, "%s: temperature must be finite and >= 0", fn);
    REQUIRE(s->draft_tokens);
    REQUIRE(s->target_logits);
    if (!greedy) REQUIRE(s->draft_logits);
    REQUIRE(s->L);
    REQUIRE(s->draft_off);
    REQUIRE(s->row_off);
    REQUIRE(s->row_req);
    REQUIRE(s->row_k);
    REQUIRE(s->accept_len);
    REQUIRE(s->num_emitted);
    REQUIRE(s->out_tokens);
    REQUIRE(s->p_tok);
    REQUIRE(s->q_tok);
    const size_t ls = dtype_size(s->logit_dtype);
    REQUIRE_ALIGNED(s->target_logits, 16);
    if (!greedy) REQUIRE_ALIGNED(s->draft_logits, 16);
    if ((size_t(s->V) * ls) % 16 != 0)
        return fail(DSPARK_EALIGN, "%s: a logit row (V=%d) is not a multiple of 16 bytes", fn, s->V);
    if (size_t(s->V) * ls > size_t(INT32_MAX))
        return fail(DSPARK_EINVAL, "%s: a logit row is too large", fn);
    // The stream work is counted in 32-bit chunk indices: at most 2^30 tiles
    // (16 TB of logits, beyond any device's memory).
    if (size_t(s->B) * size_t(s->gamma + 1) *
            ((size_t(s->V) * ls + dspark::kChunkBytes - 1) / dspark::kChunkBytes) > (size_t(1) << 30))
        return fail(DSPARK_EINVAL, "%s: B=%d gamma=%d V=%d is too large a batch", fn, s->B,
                    s->gamma, s->V);
    dspark::WorkspaceLayout lay;
    if ((st = check_workspace(s, &lay))) return st;
    DeviceInfo *dev;
    if ((st = device_info(&dev))) return st;

    const int bf = s->logit_dtype == DSPARK_BF16;
    dspark::VerifyArgs a{};
    a.B = s->B; a.gamma = s->gamma; a.V = s->V;
    a.elem_bytes = int(ls);
    a.row_bytes = int(size_t(s->V) * ls);
    a.nc = (a.row_bytes + dspark::kChunkBytes - 1) / dspark::kChunkBytes;
    a.chunk_elems = int(dspark::kChunkBytes / ls);
    a.nblk = lay.nblk;
    a.grp_stride = lay.nc;
    a.qcap = lay.qcap;
    a.qbcap = 2 * s->B;
    a.greedy = greedy;
    a.scale = greedy ? 0.f : float(1.4426950408889634 / double(s->temperature));
    a.seed = s->seed;
    a.draft_tokens = s->draft_tokens;
    a.draft_logits = s->draft_logits;
    a.target_logits = s->target_logits;
    a.L = s->L; a.draft_off = s->draft_off; a.row_off = s->row_off;
    a.row_req = s->row_req; a.row_k = s->row_k;
    a.accept_len = s->accept_len; a.num_emitted = s->num_emitted; a.out_tokens = s->out_tokens;
    a.p_tok = s->p_tok; a.q_tok = s->q_tok; a.seq_lens_commit = s->seq_lens_commit;
    a.rowrec = ws_at<float4>(s, lay.rowrec);
    a.blkrec = ws_at<float2>(s, lay.blkrec);
    a.zrec = ws_at<float2>(s, lay.zrec);
    a.gath = ws_at<float2>(s, lay.gath);
    a.dstate = ws_at<dspark::DecideState>(s, lay.dstate);
    a.q_ctr = ws_at<int32_t>(s, lay.q_ctr);
    a.req_cnt = ws_at<int32_t>(s, lay.verify_cnt);
    a.bon_cnt = ws_at<int32_t>(s, lay.bon_cnt);
    a.r1_cnt = ws_at<int32_t>(s, lay.r1_cnt);
    a.join = ws_at<int32_t>(s, lay.join);
    a.rejflag = ws_at<int32_t>(s, lay.rejflag);
    a.q_job = ws_at<int2>(s, lay.q_job);
    a.q_ready = ws_at<int32_t>(s, lay.q_ready);
    a.qb_job = ws_at<int32_t>(s, lay.qb_job);
    a.qb_ready = ws_at<int32_t>(s, lay.qb_ready);
    a.status = ws_at<int32_t>(s, lay.status);
    a.commit_len = commit_len;
    a.accept_full = accept_full;
    a.audit_totals = audit_totals;
    a.wait_ns = g_wait_ns.load();
    if (accept_full) {
        // A request with L_b = 0 has no decision rows: only its bonus draw
        // runs, so its a_b = 0 is written here.
        cudaError_t e = cudaMemsetAsync(accept_full, 0, sizeof(int32_t) * size_t(s->B),
                                        reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(accept_full)");
    }
    cudaError_t e;
    if (dspark::verify_small_fits(s->B, s->V, commit_len != nullptr)) {
        // Few requests: units of (row, 8192-id slice) over a plain grid, the
        // CTA that completes a request decides it (verify_small.cu).
        const long long units = (long long)s->B * (s->gamma + 1) * dspark::verify_small_slices(s->V);
        const int grid = int(std::min<long long>(units, (long long)dev->sms * 8));
        // Rows of four tiles or more and four requests or more: a
        // rejection's second pass goes to the tail kernel (parts over the
        // grid).  Smaller rows are cheaper in the deciding CTA than a second
        // launch, and one to three requests reject too rarely for it to pay
        // (measured: B = 8 and 16 at V = 151 936 ~10 us faster a step, B = 1
        // 1.5 us slower, V = 1024 1 us slower).
        a.small_tail = !greedy && a.nc >= 4 && s->B >= 4;
        e = dspark::launch_verify_small(a, bf, grid, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "verify_small_kernel launch");
        if (a.small_tail) {
            // The rejections' residual rows, in parts over the grid, and their
            // draws (at most one row per request, four parts each).
            const int tgrid = int(std::min<long long>((long long)s->B * 4,
                                                      (long long)dev->sms * dev->tail_blocks[bf]));
            e = dspark::launch_verify_tail(a, bf, std::max(tgrid, 1),
                                           reinterpret_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) return cuda_fail(e, "verify_tail_kernel launch");
        }
        return DSPARK_OK;
    }
    // One CTA per resident slot; the work is spread over the grid inside the
    // kernel.
    const int grid = dev->sms * dev->verify_blocks[bf];
    e = dspark::launch_verify(a, bf, grid, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "verify_kernel launch");
    return DSPARK_OK;
}

extern "C" {

dspark_status dspark_verify(const dspark_step *s, dspark_stream_t stream) {
    NvtxRange range("dspark_verify");
    return verify_impl(s, nullptr, nullptr, nullptr, stream, "dspark_verify");
}

dspark_status dspark_verify_cap_accept(const dspark_step *s, const int32_t *commit_len,
                                       int32_t *accept_full, int32_t *audit_totals,
                                       dspark_stream_t stream) {
    NvtxRange range("dspark_verify_cap_accept");
    const char *fn = "dspark_verify_cap_accept";
    if (s && s->B > 0 && !commit_len) return fail(DSPARK_EINVAL, "%s: commit_len is NULL", fn);
    return verify_impl(s, commit_len, accept_full, audit_totals, stream, fn);
}

dspark_status dspark_read_device_status(const void *workspace, int32_t *status_out,
                                        dspark_stream_t stream) {
    if (!workspace) return fail(DSPARK_EWORKSPACE, "workspace is NULL");
    if (!status_out) return fail(DSPARK_EINVAL, "status_out is NULL");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    return DSPARK_OK;
}

dspark_status dspark_set_wait_timeout_ns(uint64_t ns) {
    g_wait_ns.store(ns == 0 ? dspark::kWaitTimeoutNs : ns);
    return DSPARK_OK;
}

uint64_t dspark_wait_timeout_ns(void) { return g_wait_ns.load(); }

const char *dspark_last_error(void) { return g_err; }

const char *dspark_version(void) { return "dspark-gb300 0.1.0 (sm_103a)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// dspark_verify_noalloc: dspark_verify with its scratch in a fixed array of
// this library's device image instead of a caller workspace, for callers
// that cannot allocate device memory at the call site.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
static_assert(DSPARK_NOALLOC_SCRATCH_BYTES == kNoallocScratchBytes, "header and library agree");

// One copy per device, created when the device loads this library's module
// and held until the process exits.  In host code this name is only a
// handle: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The scratch's last kNoallocHeader bytes record the shape (B, gamma, V)
// whose counters and queue flags were last zeroed; the layout of a step uses
// the bytes before them.
constexpr size_t kNoallocHeader = 256;
constexpr size_t kNoallocLayoutBytes = kNoallocScratchBytes - kNoallocHeader;

// Per device: the array's device address.
struct NoallocSlot {
    void *ptr = nullptr;
};
NoallocSlot g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Runs on the stream before each no-alloc verify, so that the decision is
// taken on the device in stream order -- a replayed graph takes it again.
// When the shape recorded in the header differs from this call's (or reset
// is set), zero the first `need` bytes (the layout of this shape; a multiple
// of 256) and record the shape.  One CTA: the header is read before any
// thread writes.
__global__ void __launch_bounds__(1024) noalloc_prepare_kernel(unsigned char *scratch, size_t need,
                                                               int B, int gamma, int V, int reset) {
    __shared__ int s_zero;
    int *hdr = reinterpret_cast<int *>(scratch + kNoallocLayoutBytes);
    if (threadIdx.x == 0) s_zero = reset || hdr[0] != B || hdr[1] != gamma || hdr[2] != V;
    __syncthreads();
    if (!s_zero) return;
    uint4 *p = reinterpret_cast<uint4 *>(scratch);
    const size_t n16 = need / 16;
    for (size_t i = threadIdx.x; i < n16; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x == 0) {
        hdr[0] = B;
        hdr[1] = gamma;
        hdr[2] = V;
    }
}

}  // namespace

extern "C" dspark_status dspark_verify_noalloc(const dspark_step *s, int32_t reset,
                                               int32_t *status_out, dspark_stream_t stream) {
    const char *fn = "dspark_verify_noalloc";
    dspark_status st = check_shape(s);
    if (st) return st;
    const size_t need = dspark::workspace_layout(s->B, s->gamma, s->V).total;
    if (need > kNoallocLayoutBytes)
        return fail(DSPARK_EWORKSPACE,
                    "%s: B=%d gamma=%d V=%d needs %zu bytes of scratch; the static scratch holds %zu",
                    fn, s->B, s->gamma, s->V, need, kNoallocLayoutBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(DSPARK_EDEVICE, "device index %d out of range", dev);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    void *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        NoallocSlot &slot = g_noalloc[dev];
        if (!slot.ptr) {
            // First call on this device (current now): find this device's
            // copy of the array.
            e = cudaGetSymbolAddress(&slot.ptr, g_noalloc_scratch);
            if (e != cudaSuccess) {
                slot.ptr = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
            }
            if (!aligned(slot.ptr, 256)) {
                slot.ptr = nullptr;
                return fail(DSPARK_EWORKSPACE, "%s: static scratch misaligned", fn);
            }
        }
        ptr = slot.ptr;
    }
    // The counters and queue flags of this shape must start at zero.
    noalloc_prepare_kernel<<<1, 1024, 0, cs>>>(static_cast<unsigned char *>(ptr), need, s->B,
                                                 s->gamma, s->V, reset ? 1 : 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "noalloc_prepare_kernel launch");
    dspark_step local = *s;
    local.workspace = ptr;
    local.workspace_bytes = kNoallocScratchBytes;
    if ((st = dspark_verify(&local, stream))) return st;
    if (status_out) {
        const dspark::WorkspaceLayout lay = dspark::workspace_layout(s->B, s->gamma, s->V);
        e = cudaMemcpyAsync(status_out, static_cast<char *>(ptr) + lay.status, sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, cs);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(status_out)");
    }
    return DSPARK_OK;
}
