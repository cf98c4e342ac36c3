// api.cu -- the C ABI of liblachunked: argument checks, planning, dispatch.
//
// Declarations and the meaning of every argument: include/la_chunked.h.
#include <limits.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"

namespace la {

// kernels in other translation units
size_t simt_smem_bytes(int D, int dk, int fm);
int simt_inter_levels(int L, int C);
size_t simt_workspace_bytes(int B, int H, int L, int D, int dv, int C, bool loglinear);
int simt_launch(const Problem &p, int n_inter, int log2C);
bool tc_supported(const Problem &p, int num_sms);
int tc_plan(const Problem &p, int num_sms, la_plan_info *info);
int tc_launch(const Problem &p, int num_sms);
size_t nc_simt_workspace_bytes(int BH, int D, int dv);
bool nc_simt_supported(int D, int dk);
int nc_simt_launch(const Problem &p);
bool tc_nc_supported(const Problem &p);
size_t tc_nc_workspace(const Problem &p, int num_sms);
int tc_nc_launch(const Problem &p, int num_sms);
int decode_check(int B, int H, int dk, int dv, const la_feature_map *fm, int normalize,
                 int num_levels, long long t, bool loglinear, int *D_out, int *r_out);
int nc_state_launch(const Problem &p, float *S, float *z);
int state_combine_launch(float *S, float *z, const float *Sg, const float *zg, long nS, long nz, float factor,
                         cudaStream_t st);
size_t bwd_workspace_bytes(const Problem &p, int sms);
bool bwd_supported(const Problem &p);
bool bwd_tc_supported(const Problem &p, int sms);
int bwd_launch(const Problem &p, int sms, int path, const void *dout, void *dq, void *dk,
               void *dv);
int decode_launch(const void *q, const void *k, const void *v, void *out, float *S, float *z, int B,
                  int H, int dk, int dv, const la_feature_map *fm, int normalize, const float *lam,
                  int num_levels, long long t, int dtype, cudaStream_t stream,
                  float gamma);

int required_levels(int L)
{
    if (L <= 1) return 1;
    return 2 + ilog2(L - 1);
}
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x)
{
    int r = 0;
    while (x >>= 1) ++r;
    return r;
}

// ---- device error word (one per device) -------------------------------------------
__device__ int g_la_err = 0;

static int *err_ptr()
{
    static int *ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_la_err) != cudaSuccess) return nullptr;
        ptrs[dev] = (int *)p;
    }
    return ptrs[dev];
}

static int device_sms()
{
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        sms[dev] = v;
    }
    return sms[dev];
}

static bool trace_enabled()
{
    static int t = -1;
    if (t < 0) {
        const char *e = getenv("LA_TRACE");
        t = (e && *e && *e != '0') ? 1 : 0;
    }
    return t == 1;
}

// Shape / argument checks shared by every entry point; fills *p (pointers untouched).
static int check_problem(int B, int H, int L, int dk, int dv, int C, const la_feature_map *fm,
                         int normalize, bool loglinear, int num_levels, int dtype, Problem *p)
{
    if (B <= 0 || H <= 0 || L <= 0 || dk <= 0 || dv <= 0) return LA_ERR_SHAPE;
    if ((long long)B * H * L * (dk > dv ? dk : dv) > (long long)INT_MAX * 64) return LA_ERR_SHAPE;
    if ((long long)B * H > INT_MAX / 2) return LA_ERR_SHAPE;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_UNSUPPORTED;
    const int kind = fm ? fm->kind : LA_FM_IDENTITY;
    if (kind != LA_FM_IDENTITY && kind != LA_FM_ELU1 && kind != LA_FM_FAVOR)
        return LA_ERR_UNSUPPORTED;
    int D = dk;
    if (kind == LA_FM_FAVOR) {
        if (fm->m <= 0) return LA_ERR_SHAPE;
        D = fm->m;
    }
    if (D > 512 || dk > 512) return LA_ERR_UNSUPPORTED;
    // chunk size: C <= 0 means 1; C >= L means a single chunk
    if (C <= 0) C = 1;
    if (C > L) C = L;
    const int nch = (L + C - 1) / C;
    if (loglinear) {
        if (nch > 1 && !is_pow2(C)) return LA_ERR_UNSUPPORTED;
        if (num_levels < required_levels(L)) return LA_ERR_SHAPE;
    }
    memset(p, 0, sizeof(*p));
    p->B = B; p->H = H; p->L = L; p->dk = dk; p->dv = dv; p->C = C; p->D = D;
    p->fm = kind;
    p->m = (kind == LA_FM_FAVOR) ? fm->m : 0;
    p->omega = (kind == LA_FM_FAVOR) ? fm->omega : nullptr;
    p->normalize = normalize ? 1 : 0;
    p->nl = loglinear ? num_levels : 0;
    p->dtype = dtype;
    return LA_OK;
}

// Decay factor: 0 < gamma <= 1 (NaN fails the test); gamma = 1 is the plain recurrence.
static int set_decay(Problem *p, float gamma)
{
    if (!(gamma > 0.f && gamma <= 1.f)) return LA_ERR_ARG;
    p->decay = 1;
    p->gamma = gamma;
    p->l2g = (float)log2((double)gamma);
    return LA_OK;
}

static size_t simt_ws(const Problem &p, bool loglinear)
{
    return simt_workspace_bytes(p.B, p.H, p.L, p.D, p.dv, p.C, loglinear);
}

static int plan_problem(const Problem &p, bool loglinear, int path, int num_sms,
                        la_plan_info *info)
{
    memset(info, 0, sizeof(*info));
    info->chunk = p.C;
    info->n_chunks = (p.L + p.C - 1) / p.C;
    info->feature_dim = p.D;
    Problem q = p;
    if (loglinear) q.lam = (const float *)1;  // marks the log-linear mask for the planner
    if (path == LA_PATH_AUTO) path = tc_supported(q, num_sms) ? LA_PATH_TC : LA_PATH_SIMT;
    if (path == LA_PATH_TC) {
        if (!tc_supported(q, num_sms)) return LA_ERR_UNSUPPORTED;
        int rc = tc_plan(q, num_sms, info);
        info->path = LA_PATH_TC;
        return rc;
    }
    if (path != LA_PATH_SIMT) return LA_ERR_UNSUPPORTED;
    info->path = LA_PATH_SIMT;
    info->grid_x = p.B * p.H;
    info->grid_y = (p.dv + 31) / 32;
    info->block = 256;
    info->smem_bytes = (int)simt_smem_bytes(p.D, p.dk, p.fm);
    info->n_launches = 1;
    info->workspace_bytes = simt_ws(p, loglinear);
    return LA_OK;
}

static int run(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
               int dk, int dv, int C, const la_feature_map *fm, int normalize,
               const float *lam, int num_levels, int dtype, void *ws, size_t ws_bytes,
               void *stream, int path, bool decay = false, float gamma = 1.f,
               const float *S0 = nullptr, const float *z0 = nullptr, int sms_fixed = 0)
{
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    const bool ll = lam != nullptr;
    Problem p;
    int rc = check_problem(B, H, L, dk, dv, C, fm, normalize, ll, num_levels, dtype, &p);
    if (rc != LA_OK) return rc;
    if (decay && (rc = set_decay(&p, gamma)) != LA_OK) return rc;
    p.S0 = S0;
    p.z0 = z0;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    // sms_fixed = 1 keeps every head in one segment (no sequence split, no totals pass)
    const int sms = sms_fixed > 0 ? sms_fixed : device_sms();
    if (sms <= 0) return LA_ERR_CUDA;
    la_plan_info info;
    rc = plan_problem(p, ll, path, sms, &info);
    if (rc != LA_OK) return rc;
    // the tensor-core log-linear kernel copies lambda rows in bulk (16-byte aligned)
    if (info.path == LA_PATH_TC && ll && ((uintptr_t)lam & 15) != 0) {
        if (path != LA_PATH_AUTO) return LA_ERR_UNSUPPORTED;
        rc = plan_problem(p, ll, LA_PATH_SIMT, sms, &info);
        if (rc != LA_OK) return rc;
    }
    if (info.workspace_bytes > 0 && (!ws || ws_bytes < info.workspace_bytes))
        return LA_ERR_WORKSPACE;
    p.q = q; p.k = k; p.v = v; p.out = out;
    p.lam = lam;
    p.workspace = ws;
    p.workspace_bytes = ws_bytes;
    p.stream = (cudaStream_t)stream;
    p.err = err_ptr();
    if (!p.err) return LA_ERR_CUDA;
    if (trace_enabled())
        fprintf(stderr,
                "[la] B=%d H=%d L=%d dk=%d dv=%d C=%d D=%d fm=%d norm=%d ll=%d gamma=%g dtype=%d -> "
                "path=%d grid=(%d,%d) block=%d smem=%d ws=%zu launches=%d\n",
                B, H, L, dk, dv, p.C, p.D, p.fm, p.normalize, (int)ll, decay ? gamma : 1.0, dtype, info.path,
                info.grid_x, info.grid_y, info.block, info.smem_bytes, info.workspace_bytes,
                info.n_launches);
    if (info.path == LA_PATH_TC) return tc_launch(p, sms);
    int log2C = ll ? ilog2(p.C) : 0;
    int n_inter = ll ? simt_inter_levels(p.L, p.C) : 0;
    return simt_launch(p, n_inter, log2C);
}

}  // namespace la

using namespace la;

extern "C" {

int la_chunked_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                   int dk, int dv, int C, const la_feature_map *feature_map, int normalize,
                   const float *level_weights, int num_levels, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream)
{
    return run(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, level_weights,
               num_levels, dtype, workspace, workspace_bytes, stream, LA_PATH_AUTO);
}

int la_chunked_fwd_path(const void *q, const void *k, const void *v, void *out, int B, int H,
                        int L, int dk, int dv, int C, const la_feature_map *feature_map,
                        int normalize, const float *level_weights, int num_levels, int dtype,
                        void *workspace, size_t workspace_bytes, void *stream, int path)
{
    return run(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, level_weights,
               num_levels, dtype, workspace, workspace_bytes, stream, path);
}

int la_chunked_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                        void *out_host, void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                        int B, int H, int L, int dk, int dv, int C,
                        const la_feature_map *feature_map, int normalize,
                        const float *level_weights, int num_levels, int dtype, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    if (!q_host || !k_host || !v_host || !out_host) return LA_ERR_NULL;
    if (!q_dev || !k_dev || !v_dev || !out_dev) return LA_ERR_NULL;
    Problem p;
    const bool ll = level_weights != nullptr;
    int rc = check_problem(B, H, L, dk, dv, C, feature_map, normalize, ll, num_levels, dtype, &p);
    if (rc != LA_OK) return rc;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    const int sms = device_sms();
    if (sms <= 0) return LA_ERR_CUDA;
    la_plan_info info;
    if ((rc = plan_problem(p, ll, LA_PATH_AUTO, sms, &info)) != LA_OK) return rc;
    // as in run(): level weights that are not 16-byte aligned take the generic path
    if (info.path == LA_PATH_TC && ll && ((uintptr_t)level_weights & 15) != 0 &&
        (rc = plan_problem(p, ll, LA_PATH_SIMT, sms, &info)) != LA_OK)
        return rc;
    if (info.workspace_bytes > 0 && (!workspace || workspace_bytes < info.workspace_bytes))
        return LA_ERR_WORKSPACE;
    const size_t es = dtype == LA_F32 ? 4 : 2;
    const int BH = B * H;
    const size_t hqk = (size_t)L * dk * es, hv = (size_t)L * dv * es;  // bytes per head
    cudaStream_t s = (cudaStream_t)stream;
    // Pipelined over groups of heads when the plan is one unsplit launch and the step moves
    // enough bytes: the copies in of group i+1 and out of group i-1 run on their own streams
    // (the two copy directions at once) while group i computes.  Every group runs unsplit,
    // so each head gets exactly the arithmetic of the whole launch.
    int ng = 1;
    if (info.n_launches == 1 && (size_t)BH * 2 * (hqk + hv) >= ((size_t)64 << 20)) ng = BH < 8 ? BH : 8;
    const int hg = (BH + ng - 1) / ng;
    ng = (BH + hg - 1) / hg;
    if (ng > 1) {
        // every group runs on the whole problem's path with a workspace that fits it; a
        // group's level weights start 16-byte aligned when the whole array does
        Problem pg;
        la_plan_info gi;
        if (check_problem(1, hg, L, dk, dv, C, feature_map, normalize, ll, num_levels, dtype, &pg) != LA_OK ||
            plan_problem(pg, ll, info.path, 1, &gi) != LA_OK || gi.path != info.path ||
            (gi.workspace_bytes > 0 && (!workspace || workspace_bytes < gi.workspace_bytes)) ||
            (ll && ((size_t)hg * L * num_levels) % 4 != 0))
            ng = 1;
    }
    if (ng == 1) {
        if (cudaMemcpyAsync(q_dev, q_host, BH * hqk, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(k_dev, k_host, BH * hqk, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(v_dev, v_host, BH * hv, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return LA_ERR_CUDA;
        rc = la_chunked_fwd(q_dev, k_dev, v_dev, out_dev, B, H, L, dk, dv, C, feature_map,
                            normalize, level_weights, num_levels, dtype, workspace, workspace_bytes,
                            stream);
        if (rc != LA_OK) return rc;
        if (cudaMemcpyAsync(out_host, out_dev, BH * hv, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return LA_ERR_CUDA;
        return LA_OK;
    }
    // streams and events of this call (released once their work completes)
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t ev[2 * 8 + 3] = {};
    const int nev = 2 * ng + 3;
    bool ok = cudaStreamCreateWithFlags(&cin, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&cout, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < nev; ++i)
        ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    cudaEvent_t start = ev[0], done = ev[1];
    // both copy streams start after the work already queued on the caller's stream
    ok = ok && cudaEventRecord(start, s) == cudaSuccess && cudaStreamWaitEvent(cin, start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(cout, start, 0) == cudaSuccess;
    rc = ok ? LA_OK : LA_ERR_CUDA;
    auto at = [](const void *base, size_t off) { return (void *)((const char *)base + off); };
    for (int g = 0; rc == LA_OK && g < ng; ++g) {
        const int h0 = g * hg, hn = BH - h0 < hg ? BH - h0 : hg;
        cudaEvent_t in_done = ev[2 + 2 * g], run_done = ev[3 + 2 * g];
        const size_t oqk = (size_t)h0 * hqk, ov = (size_t)h0 * hv;
        if (cudaMemcpyAsync(at(q_dev, oqk), at(q_host, oqk), hn * hqk, cudaMemcpyHostToDevice, cin) != cudaSuccess ||
            cudaMemcpyAsync(at(k_dev, oqk), at(k_host, oqk), hn * hqk, cudaMemcpyHostToDevice, cin) != cudaSuccess ||
            cudaMemcpyAsync(at(v_dev, ov), at(v_host, ov), hn * hv, cudaMemcpyHostToDevice, cin) != cudaSuccess ||
            cudaEventRecord(in_done, cin) != cudaSuccess || cudaStreamWaitEvent(s, in_done, 0) != cudaSuccess) {
            rc = LA_ERR_CUDA;
            break;
        }
        const float *lam = ll ? level_weights + (size_t)h0 * L * num_levels : nullptr;
        rc = run(at(q_dev, oqk), at(k_dev, oqk), at(v_dev, ov), at(out_dev, ov), 1, hn, L, dk, dv, C,
                 feature_map, normalize, lam, num_levels, dtype, workspace, workspace_bytes, stream,
                 info.path, false, 1.f, nullptr, nullptr, 1);
        if (rc != LA_OK) break;
        if (cudaEventRecord(run_done, s) != cudaSuccess || cudaStreamWaitEvent(cout, run_done, 0) != cudaSuccess ||
            cudaMemcpyAsync(at(out_host, ov), at(out_dev, ov), hn * hv, cudaMemcpyDeviceToHost, cout) != cudaSuccess)
            rc = LA_ERR_CUDA;
    }
    // the caller's stream reaches the end of the call after every copy of both streams,
    // also when a group failed to queue (nothing is left running past the call)
    cudaEvent_t in_end = ev[nev - 1];
    if (done && in_end && cin && cout) {
        if (cudaEventRecord(in_end, cin) != cudaSuccess || cudaStreamWaitEvent(s, in_end, 0) != cudaSuccess ||
            cudaEventRecord(done, cout) != cudaSuccess || cudaStreamWaitEvent(s, done, 0) != cudaSuccess)
            if (rc == LA_OK) rc = LA_ERR_CUDA;
    }
    for (int i = 0; i < nev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    if (cin) cudaStreamDestroy(cin);
    if (cout) cudaStreamDestroy(cout);
    return rc;
}

size_t la_chunked_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                  const la_feature_map *feature_map, int normalize,
                                  int num_levels, int dtype)
{
    Problem p;
    const bool ll = num_levels > 0;
    if (check_problem(B, H, L, dk, dv, C, feature_map, normalize, ll, num_levels, dtype, &p) !=
        LA_OK)
        return 0;
    const int sms = device_sms();
    la_plan_info info;
    if (plan_problem(p, ll, LA_PATH_AUTO, sms > 0 ? sms : 152, &info) != LA_OK) return 0;
    // enough for either path, so a caller may force a path with the same buffer
    size_t a = info.workspace_bytes, b = simt_ws(p, ll);
    return a > b ? a : b;
}

int la_chunked_plan(int B, int H, int L, int dk, int dv, int C,
                    const la_feature_map *feature_map, int normalize, int loglinear,
                    int num_levels, int dtype, int path, int num_sms, la_plan_info *info)
{
    if (!info) return LA_ERR_NULL;
    Problem p;
    int rc = check_problem(B, H, L, dk, dv, C, feature_map, normalize, loglinear != 0,
                           num_levels, dtype, &p);
    if (rc != LA_OK) return rc;
    if (num_sms <= 0) num_sms = device_sms();
    if (num_sms <= 0) return LA_ERR_CUDA;
    return plan_problem(p, loglinear != 0, path, num_sms, info);
}

int la_last_device_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    int *ep = err_ptr();
    if (!ep) return LA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, ep, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    if (h != 0) {
        const int zero = 0;
        if (cudaMemcpy(ep, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return LA_ERR_CUDA;
    }
    return h;
}

const char *la_status_string(int status)
{
    switch (status) {
    case LA_OK: return "ok";
    case LA_ERR_NULL: return "a required pointer is NULL";
    case LA_ERR_SHAPE: return "invalid or inconsistent sizes";
    case LA_ERR_UNSUPPORTED: return "unsupported combination of dtype, sizes, feature map or C";
    case LA_ERR_WORKSPACE: return "workspace missing or too small";
    case LA_ERR_CUDA: return "a CUDA runtime call failed";
    case LA_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case LA_ERR_DEVICE: return "a device-side check failed";
    case LA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed no-alloc buffer (8 MiB) holds";
    case LA_ERR_ARG: return "an argument value is out of range";
    default: return "unknown status";
    }
}

int la_cost_model(long long L, long long D, long long C, long long *state_macs,
                  long long *score_macs)
{
    if (L < 0 || D < 0 || C < 0) return LA_ERR_SHAPE;
    // "attention と線形の間", section 3: per chunk, writing and reading the state cost
    // C D^2 each (L/C chunks -> 2 L D^2); making the scores and mixing the values cost
    // C^2 D each (-> 2 L C D).
    if (state_macs) *state_macs = 2 * L * D * D;
    if (score_macs) *score_macs = 2 * L * C * D;
    return LA_OK;
}

int la_decode_step(const void *q, const void *k, const void *v, void *out, float *state,
                   float *zstate, int B, int H, int dk, int dv,
                   const la_feature_map *feature_map, int normalize,
                   const float *level_weights, int num_levels, long long t, int dtype,
                   void *stream)
{
    if (!q || !k || !v || !out || !state) return LA_ERR_NULL;
    if (normalize && !zstate) return LA_ERR_NULL;
    if ((long long)B * H > INT_MAX / 2) return LA_ERR_SHAPE;
    return decode_launch(q, k, v, out, state, zstate, B, H, dk, dv, feature_map, normalize,
                         level_weights, num_levels, t, dtype, (cudaStream_t)stream, 1.f);
}

int la_decay_decode_step(const void *q, const void *k, const void *v, void *out, float *state,
                         float *zstate, int B, int H, int dk, int dv,
                         const la_feature_map *feature_map, int normalize, float gamma,
                         int dtype, void *stream)
{
    if (!q || !k || !v || !out || !state) return LA_ERR_NULL;
    if (normalize && !zstate) return LA_ERR_NULL;
    if ((long long)B * H > INT_MAX / 2) return LA_ERR_SHAPE;
    if (!(gamma > 0.f && gamma <= 1.f)) return LA_ERR_ARG;
    return decode_launch(q, k, v, out, state, zstate, B, H, dk, dv, feature_map, normalize,
                         nullptr, 0, 0, dtype, (cudaStream_t)stream, gamma);
}

long long la_decode_state_elems(int B, int H, int dk, int dv, const la_feature_map *feature_map,
                                int num_levels, long long *z_elems)
{
    int D = 0, r = 0;
    const bool ll = num_levels > 0;
    if (decode_check(B, H, dk, dv, feature_map, 0, ll ? num_levels : 0, 0, ll, &D, &r) != LA_OK) {
        if (z_elems) *z_elems = 0;
        return 0;
    }
    const long long lv = ll ? num_levels - 1 : 1;
    if (z_elems) *z_elems = (long long)B * H * lv * D;
    return (long long)B * H * lv * D * dv;
}

// non-causal: one global state per head; the tensor-core path when it covers the shape
static int nc_problem(int B, int H, int L, int dk, int dv, const la_feature_map *fm, int normalize,
                      int dtype, Problem *p)
{
    int rc = check_problem(B, H, L, dk, dv, 64, fm, normalize, false, 0, dtype, p);
    if (rc != LA_OK) return rc;
    if (!nc_simt_supported(p->D, p->dk)) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

size_t la_noncausal_workspace_bytes(int B, int H, int L, int dk, int dv,
                                    const la_feature_map *feature_map, int normalize, int dtype)
{
    Problem p;
    if (nc_problem(B, H, L, dk, dv, feature_map, normalize, dtype, &p) != LA_OK) return 0;
    const int sms = device_sms();
    size_t a = nc_simt_workspace_bytes(B * H, p.D, dv);
    size_t b = tc_nc_supported(p) ? tc_nc_workspace(p, sms > 0 ? sms : 152) : 0;
    return a > b ? a : b;
}

int la_noncausal_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                     int dk, int dv, const la_feature_map *feature_map, int normalize, int dtype,
                     void *workspace, size_t workspace_bytes, void *stream)
{
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    Problem p;
    int rc = nc_problem(B, H, L, dk, dv, feature_map, normalize, dtype, &p);
    if (rc != LA_OK) return rc;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    const int sms = device_sms();
    if (sms <= 0) return LA_ERR_CUDA;
    const bool tc = tc_nc_supported(p);
    const size_t need = tc ? tc_nc_workspace(p, sms) : nc_simt_workspace_bytes(B * H, p.D, dv);
    if (!workspace || workspace_bytes < need) return LA_ERR_WORKSPACE;
    p.q = q; p.k = k; p.v = v; p.out = out;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    p.stream = (cudaStream_t)stream;
    p.err = err_ptr();
    if (!p.err) return LA_ERR_CUDA;
    return tc ? tc_nc_launch(p, sms) : nc_simt_launch(p);
}

// ---- decay (Retention)
int la_decay_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                 int dk, int dv, int C, const la_feature_map *feature_map, int normalize,
                 float gamma, int dtype, void *workspace, size_t workspace_bytes, void *stream,
                 int path)
{
    return run(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, nullptr, 0, dtype,
               workspace, workspace_bytes, stream, path, true, gamma);
}

size_t la_decay_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                const la_feature_map *feature_map, int normalize, float gamma,
                                int dtype)
{
    Problem p;
    if (check_problem(B, H, L, dk, dv, C, feature_map, normalize, false, 0, dtype, &p) != LA_OK ||
        set_decay(&p, gamma) != LA_OK)
        return 0;
    const int sms = device_sms();
    la_plan_info info;
    if (plan_problem(p, false, LA_PATH_AUTO, sms > 0 ? sms : 152, &info) != LA_OK) return 0;
    return info.workspace_bytes;  // the generic path needs none
}

int la_decay_plan(int B, int H, int L, int dk, int dv, int C, const la_feature_map *feature_map,
                  int normalize, float gamma, int dtype, int path, int num_sms, la_plan_info *info)
{
    if (!info) return LA_ERR_NULL;
    Problem p;
    int rc = check_problem(B, H, L, dk, dv, C, feature_map, normalize, false, 0, dtype, &p);
    if (rc != LA_OK) return rc;
    if ((rc = set_decay(&p, gamma)) != LA_OK) return rc;
    if (num_sms <= 0) num_sms = device_sms();
    if (num_sms <= 0) return LA_ERR_CUDA;
    return plan_problem(p, false, path, num_sms, info);
}

// ---- backward pass
static int bwd_problem(int B, int H, int L, int dk, int dv, int C, const la_feature_map *fm,
                       int normalize, float gamma, int dtype, Problem *p)
{
    int rc = check_problem(B, H, L, dk, dv, C, fm, normalize, false, 0, dtype, p);
    if (rc != LA_OK) return rc;
    if (gamma != 1.f && (rc = set_decay(p, gamma)) != LA_OK) return rc;
    if (!bwd_supported(*p)) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

size_t la_chunked_bwd_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                      const la_feature_map *feature_map, int normalize,
                                      int dtype)
{
    Problem p;
    if (bwd_problem(B, H, L, dk, dv, C, feature_map, normalize, 1.f, dtype, &p) != LA_OK) return 0;
    const int sms = device_sms();
    return bwd_workspace_bytes(p, sms > 0 ? sms : 152);
}

int la_chunked_bwd(const void *q, const void *k, const void *v, const void *dout, void *dq,
                   void *dk_, void *dv_, int B, int H, int L, int dk,
                   int dv, int C, const la_feature_map *feature_map, int normalize, float gamma,
                   int dtype, void *workspace, size_t workspace_bytes, void *stream, int path)
{
    if (!q || !k || !v || !dout || !dq || !dk_ || !dv_) return LA_ERR_NULL;
    Problem p;
    int rc = bwd_problem(B, H, L, dk, dv, C, feature_map, normalize, gamma, dtype, &p);
    if (rc != LA_OK) return rc;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    if (path != LA_PATH_AUTO && path != LA_PATH_SIMT && path != LA_PATH_TC) return LA_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return LA_ERR_CUDA;
    if (!workspace || workspace_bytes < bwd_workspace_bytes(p, sms)) return LA_ERR_WORKSPACE;
    p.q = q; p.k = k; p.v = v;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    p.stream = (cudaStream_t)stream;
    p.err = err_ptr();
    if (!p.err) return LA_ERR_CUDA;
    return bwd_launch(p, sms, path, dout, dq, dk_, dv_);
}

// ---- backward pass under the log-linear mask (generic route)
static int bwd_ll_problem(int B, int H, int L, int dk, int dv, int C, const la_feature_map *fm,
                          int normalize, int num_levels, int dtype, Problem *p)
{
    int rc = check_problem(B, H, L, dk, dv, C, fm, normalize, true, num_levels, dtype, p);
    if (rc != LA_OK) return rc;
    p->lam = (const float *)1;  // marks the mask for the support check; set to the caller's below
    if (!bwd_supported(*p)) return LA_ERR_UNSUPPORTED;
    p->lam = nullptr;
    return LA_OK;
}

size_t la_chunked_bwd_ll_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                         const la_feature_map *feature_map, int normalize,
                                         int num_levels, int dtype)
{
    Problem p;
    if (bwd_ll_problem(B, H, L, dk, dv, C, feature_map, normalize, num_levels, dtype, &p) != LA_OK) return 0;
    p.lam = (const float *)256;  // a 16-byte aligned stand-in: the size is that of aligned weights
    const int sms = device_sms();
    return bwd_workspace_bytes(p, sms > 0 ? sms : 152);
}

int la_chunked_bwd_ll(const void *q, const void *k, const void *v, const void *dout, void *dq,
                      void *dk_, void *dv_, int B, int H, int L, int dk, int dv, int C,
                      const la_feature_map *feature_map, int normalize, const float *level_weights,
                      int num_levels, int dtype, void *workspace, size_t workspace_bytes, void *stream,
                      int path)
{
    if (!q || !k || !v || !dout || !dq || !dk_ || !dv_ || !level_weights) return LA_ERR_NULL;
    Problem p;
    int rc = bwd_ll_problem(B, H, L, dk, dv, C, feature_map, normalize, num_levels, dtype, &p);
    if (rc != LA_OK) return rc;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    if (path == LA_PATH_TC) return LA_ERR_UNSUPPORTED;
    if (path != LA_PATH_AUTO && path != LA_PATH_SIMT) return LA_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return LA_ERR_CUDA;
    p.lam = level_weights;
    if (!workspace || workspace_bytes < bwd_workspace_bytes(p, sms)) return LA_ERR_WORKSPACE;
    p.q = q; p.k = k; p.v = v;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    p.stream = (cudaStream_t)stream;
    p.err = err_ptr();
    if (!p.err) return LA_ERR_CUDA;
    return bwd_launch(p, sms, LA_PATH_SIMT, dout, dq, dk_, dv_);
}

// ---- carried state: final state of a pass, combining segment states, a pass from a state
int la_chunked_state(const void *k, const void *v, float *state, float *zstate, int B, int H, int L,
                     int dk, int dv, const la_feature_map *feature_map, float gamma, int dtype,
                     void *stream)
{
    if (!k || !v || !state) return LA_ERR_NULL;
    Problem p;
    int rc = check_problem(B, H, L, dk, dv, 1, feature_map, zstate != nullptr, false, 0, dtype, &p);
    if (rc != LA_OK) return rc;
    if (gamma != 1.f && (rc = set_decay(&p, gamma)) != LA_OK) return rc;
    if (p.fm == LA_FM_FAVOR && !p.omega) return LA_ERR_NULL;
    p.k = k;
    p.v = v;
    p.stream = (cudaStream_t)stream;
    return nc_state_launch(p, state, zstate);
}

int la_state_combine(float *state, float *zstate, const float *seg_state, const float *seg_zstate,
                     int B, int H, int D, int dv, float factor, void *stream)
{
    if (!state || !seg_state) return LA_ERR_NULL;
    if ((zstate == nullptr) != (seg_zstate == nullptr)) return LA_ERR_NULL;
    if (B <= 0 || H <= 0 || D <= 0 || dv <= 0) return LA_ERR_SHAPE;
    if (!(factor >= 0.f && factor <= 1.f)) return LA_ERR_ARG;
    const long nS = (long)B * H * D * dv, nz = zstate ? (long)B * H * D : 0;
    return state_combine_launch(state, zstate, seg_state, seg_zstate, nS, nz, factor,
                                (cudaStream_t)stream);
}

int la_chunked_fwd_init(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                        int dk, int dv, int C, const la_feature_map *feature_map, int normalize,
                        float gamma, const float *state0, const float *zstate0, int dtype,
                        void *workspace, size_t workspace_bytes, void *stream, int path)
{
    return run(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, nullptr, 0, dtype,
               workspace, workspace_bytes, stream, path, gamma != 1.f, gamma, state0, zstate0);
}

const char *la_version(void) { return "0.1.0"; }

}  // extern "C"
