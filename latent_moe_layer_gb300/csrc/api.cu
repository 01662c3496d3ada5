// C ABI: handle lifecycle, weight checks, workspace layout and the forward
// orchestration on the caller's stream.
#include <new>
#include <string.h>

#include "k3moe_internal.h"
#include "tc.h"

using namespace k3;

thread_local long g_k3_launches = 0;

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Carver {
    uint8_t *base;
    size_t off = 0;
    template <class T>
    T *take(size_t count)
    {
        off = align_up(off, 256);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += sizeof(T) * count;
        return p;
    }
};

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return na && nb && x < y + nb && y < x + na;
}

// Scan scale bytes for 255 (E8M0 NaN): grid (n_groups, 6 matrices).
__global__ void scan_scales_kernel(const uint8_t *const *tabs0, const uint8_t *const *tabs1,
                                   const uint8_t *const *tabs2, size_t n0, size_t n2, int *flag)
{
    const uint8_t *p;
    size_t n;
    if (blockIdx.y == 0) { p = tabs0[blockIdx.x]; n = n0; }
    else if (blockIdx.y == 1) { p = tabs1[blockIdx.x]; n = n0; }
    else { p = tabs2[blockIdx.x]; n = n2; }
    int bad = 0;
    for (size_t i = threadIdx.x; i < n; i += blockDim.x) bad |= (p[i] == 255);
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(flag, 1);
}

__global__ void scan_bytes_kernel(const uint8_t *p, size_t n, int *flag)
{
    int bad = 0;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        bad |= (p[i] == 255);
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(flag, 1);
}

size_t persistent_layout(const k3moe_config &c, uint8_t *base, k3moe_handle *h)
{
    Carver cv{base};
    int *st = cv.take<int>(ST_COUNT);
    const uint8_t **tabs[6];
    for (int i = 0; i < 6; ++i) tabs[i] = cv.take<const uint8_t *>(c.n_experts);
    const uint8_t **shtab = cv.take<const uint8_t *>(6);
    size_t ntm = k3_tc_tmap_count(c);
    void *tm = cv.take<uint8_t>(ntm * 128 + 128);
    uint8_t *rmax = cv.take<uint8_t>(k3_tc_rowmax_bytes(c));
    uint16_t *hilo = cv.take<uint16_t>(k3_tc_hilo_bytes(c) / 2 + 1);
    int *flag = cv.take<int>(1);
    (void)flag;
    float *glu_bound = cv.take<float>(4);
    // one counter per 128-row output tile of the decode-size dense GEMMs
    const int cnt_up = (c.n_experts + 127) / 128 + (c.latent + 127) / 128;
    const int cnt_n = cnt_up + (c.hidden + 127) / 128;
    int *dcnt = cv.take<int>(cnt_n);
    if (h) {
        h->d_dense_cnt = dcnt;
        h->dense_cnt_up = cnt_up;
        h->dense_cnt_n = cnt_n;
        h->d_status = st;
        for (int i = 0; i < 6; ++i) h->d_eptr[i] = tabs[i];
        h->d_shtab = shtab;
        h->d_tmaps = base ? (void *)align_up((uintptr_t)tm, 128) : nullptr;
        h->tmap_count = ntm;
        h->d_rowmax = rmax;
        h->d_router_hilo = hilo;
        h->d_glu_bound = glu_bound;
    }
    return align_up(cv.off, 256);
}

}  // namespace

extern "C" {

const char *k3moe_strerror(int code)
{
    switch (code) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_ARG: return "invalid argument";
    case K3MOE_ERR_SHAPE: return "unsupported shape";
    case K3MOE_ERR_ALIGN: return "pointer or row not 16-byte aligned";
    case K3MOE_ERR_BAD_SCALE: return "E8M0 scale byte 255 (NaN)";
    case K3MOE_ERR_ALIAS: return "output overlaps input";
    case K3MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case K3MOE_ERR_CUDA: return "CUDA call failed";
    case K3MOE_ERR_TIMEOUT: return "device wait timed out";
    case K3MOE_ERR_UNSUPPORTED: return "unsupported option";
    case K3MOE_ERR_RANGE: return "expert index out of range or f16 overflow";
    case K3MOE_ERR_STATE: return "call out of order";
    default: return "unknown error";
    }
}

int k3moe_create(const k3moe_config *cfg, k3moe_handle **out)
{
    if (!cfg || !out) return K3MOE_ERR_ARG;
    const k3moe_config &c = *cfg;
    if (c.hidden <= 0 || c.latent <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.inter <= 0 ||
        c.shared_inter < 0)
        return K3MOE_ERR_ARG;
    if (c.hidden % 32 || c.latent % 32 || c.inter % 32 || c.shared_inter % 32) return K3MOE_ERR_SHAPE;
    if (c.n_experts > 1024 || c.top_k > 32 || c.top_k > c.n_experts) return K3MOE_ERR_SHAPE;
    if (c.latent > 8192) return K3MOE_ERR_SHAPE;
    if (c.act != K3MOE_ACT_SILU && c.act != K3MOE_ACT_SITU) return K3MOE_ERR_UNSUPPORTED;
    if (!(c.situ_beta == c.situ_beta) || !(c.situ_linear_beta == c.situ_linear_beta)) return K3MOE_ERR_ARG;
    if (c.a8 != 0 && c.a8 != 1) return K3MOE_ERR_ARG;
    if (c.router_dtype != K3MOE_ROUTER_F32 && c.router_dtype != K3MOE_ROUTER_BF16) return K3MOE_ERR_ARG;
    if (c.path < K3MOE_PATH_AUTO || c.path > K3MOE_PATH_TENSOR) return K3MOE_ERR_ARG;
    if (!(c.rms_eps >= 0.f) || !(c.routed_scaling == c.routed_scaling)) return K3MOE_ERR_ARG;
    k3moe_handle *h = new (std::nothrow) k3moe_handle();
    if (!h) return K3MOE_ERR_ARG;
    h->cfg = c;
    if (!(h->cfg.situ_beta > 0.f)) h->cfg.situ_beta = 4.0f;                 // the released config's values
    if (!(h->cfg.situ_linear_beta > 0.f)) h->cfg.situ_linear_beta = 25.0f;
    *out = h;
    return K3MOE_OK;
}

static void prof_free(k3moe_handle *h)
{
    if (!h->prof) return;
    for (int r = 0; r < k3_prof::RING; ++r)
        for (int s = 0; s < K3MOE_NUM_STAGES; ++s)
            for (int q = 0; q < 2; ++q) cudaEventDestroy(h->prof->ev[r][s][q]);
    delete h->prof;
    h->prof = nullptr;
}

void k3moe_destroy(k3moe_handle *h)
{
    if (!h) return;
    prof_free(h);
    delete h;
}

int k3moe_profile_enable(k3moe_handle *h, int enable)
{
    if (!h) return K3MOE_ERR_ARG;
    if (!enable) {
        prof_free(h);
        return K3MOE_OK;
    }
    if (h->prof) return K3MOE_OK;
    k3_prof *p = new (std::nothrow) k3_prof();
    if (!p) return K3MOE_ERR_ARG;
    for (int r = 0; r < k3_prof::RING; ++r)
        for (int s = 0; s < K3MOE_NUM_STAGES; ++s) {
            p->used[r][s] = false;
            for (int q = 0; q < 2; ++q)
                if (cudaEventCreate(&p->ev[r][s][q]) != cudaSuccess) return K3MOE_ERR_CUDA;
        }
    for (int s = 0; s < K3MOE_NUM_STAGES; ++s) p->launches[s] = 0;
    p->on = true;
    h->prof = p;
    return K3MOE_OK;
}

int k3moe_profile_read(k3moe_handle *h, float *stage_ms, int *stage_launches, cudaStream_t st)
{
    if (!h || !stage_ms) return K3MOE_ERR_ARG;
    if (!h->prof) return K3MOE_ERR_STATE;
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    k3_prof *p = h->prof;
    for (int s = 0; s < K3MOE_NUM_STAGES; ++s) {
        double acc = 0.0;
        for (int r = 0; r < p->pos; ++r)
            if (p->used[r][s]) {
                float ms = 0.f;
                K3_CUDA_TRY(cudaEventElapsedTime(&ms, p->ev[r][s][0], p->ev[r][s][1]));
                acc += ms;
                p->used[r][s] = false;
            }
        stage_ms[s] = (float)acc;
        if (stage_launches) stage_launches[s] = (int)p->launches[s];
        p->launches[s] = 0;
    }
    int n = p->pos;
    p->pos = 0;
    return n;
}

const char *k3moe_stage_name(int s)
{
    static const char *names[K3MOE_NUM_STAGES] = {"router", "down_proj", "topk", "permute", "gate_up",
                                                  "expert_down", "combine_norm", "up_proj", "shared",
                                                  "finish", "prep", "shared_down"};
    return (s >= 0 && s < K3MOE_NUM_STAGES) ? names[s] : "?";
}

size_t k3moe_persistent_bytes(const k3moe_handle *h)
{
    if (!h) return 0;
    return persistent_layout(h->cfg, nullptr, nullptr);
}

int k3moe_load_weights(k3moe_handle *h, const k3moe_weights *w, void *persistent,
                       size_t persistent_bytes, cudaStream_t st)
{
    if (!h || !w || !persistent) return K3MOE_ERR_ARG;
    const k3moe_config &c = h->cfg;
    if (persistent_bytes < k3moe_persistent_bytes(h)) return K3MOE_ERR_WORKSPACE;
    if ((uintptr_t)persistent % 256) return K3MOE_ERR_ALIGN;
    if (!w->w_router || !w->w_down || !w->w_up || !w->norm_gamma) return K3MOE_ERR_ARG;
    if (c.has_select_bias && !w->select_bias) return K3MOE_ERR_ARG;
    const uint8_t *const *tabs[6] = {w->w1_packed, w->w1_scale, w->w3_packed,
                                     w->w3_scale, w->w2_packed, w->w2_scale};
    for (int i = 0; i < 6; ++i) {
        if (!tabs[i]) return K3MOE_ERR_ARG;
        for (int e = 0; e < c.n_experts; ++e)
            if (!tabs[i][e]) return K3MOE_ERR_ARG;
    }
    const uint8_t *sh[6] = {w->ws1_packed, w->ws1_scale, w->ws3_packed,
                            w->ws3_scale, w->ws2_packed, w->ws2_scale};
    if (c.shared_inter > 0)
        for (int i = 0; i < 6; ++i)
            if (!sh[i]) return K3MOE_ERR_ARG;

    // 16-byte alignment of every packed/scale row (tensor path requirement)
    // (tensor path: K of every GEMM a multiple of 512 = 16-byte scale groups, rows a multiple of 128)
    bool al = c.latent % 512 == 0 && c.inter % 512 == 0 && c.hidden % 128 == 0;
    for (int i = 0; i < 6 && al; ++i)
        for (int e = 0; e < c.n_experts; ++e)
            if ((uintptr_t)tabs[i][e] % 16) { al = false; break; }
    if (c.shared_inter > 0) {
        al = al && c.hidden % 512 == 0 && c.shared_inter % 512 == 0;
        for (int i = 0; i < 6; ++i) al = al && ((uintptr_t)sh[i] % 16 == 0);
    }
    // A8: the block-scaled expert GEMMs read the packed FP4 rows through TMA's
    // unpacking type, which needs 32-byte aligned bases and row strides
    if (c.a8) {
        al = al && c.latent % 64 == 0 && c.inter % 64 == 0;
        for (int i = 0; i < 6 && al; i += 2)
            for (int e = 0; e < c.n_experts; ++e)
                if ((uintptr_t)tabs[i][e] % 32) { al = false; break; }
    }
    if (c.path == K3MOE_PATH_TENSOR && !al) return K3MOE_ERR_ALIGN;

    K3_CUDA_TRY(cudaGetDevice(&h->device));
    K3_CUDA_TRY(cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
    h->persist = (uint8_t *)persistent;
    h->persist_bytes = persistent_bytes;
    persistent_layout(c, h->persist, h);
    K3_CUDA_TRY(cudaMemsetAsync(h->d_status, 0, sizeof(int) * ST_COUNT, st));
    K3_CUDA_TRY(cudaMemsetAsync(h->d_dense_cnt, 0, sizeof(int) * h->dense_cnt_n, st));
    for (int i = 0; i < 6; ++i)
        K3_CUDA_TRY(cudaMemcpyAsync((void *)h->d_eptr[i], tabs[i], sizeof(void *) * c.n_experts,
                                    cudaMemcpyHostToDevice, st));
    K3_CUDA_TRY(cudaMemcpyAsync((void *)h->d_shtab, sh, sizeof(void *) * 6, cudaMemcpyHostToDevice, st));
    // scale scan (E8M0 255 is NaN: rejected)
    int *flag = h->d_status + 2;
    K3_CUDA_TRY(cudaMemsetAsync(flag, 0, sizeof(int), st));
    scan_scales_kernel<<<dim3(c.n_experts, 3), 256, 0, st>>>(
        h->d_eptr[1], h->d_eptr[3], h->d_eptr[5], (size_t)c.inter * (c.latent / 32),
        (size_t)c.latent * (c.inter / 32), flag);
    if (c.shared_inter > 0) {
        scan_bytes_kernel<<<64, 256, 0, st>>>(sh[1], (size_t)c.shared_inter * (c.hidden / 32), flag);
        scan_bytes_kernel<<<64, 256, 0, st>>>(sh[3], (size_t)c.shared_inter * (c.hidden / 32), flag);
        scan_bytes_kernel<<<64, 256, 0, st>>>(sh[5], (size_t)c.hidden * (c.shared_inter / 32), flag);
    }
    K3_CUDA_TRY(cudaGetLastError());
    int bad = 0;
    K3_CUDA_TRY(cudaMemcpyAsync(&bad, flag, sizeof(int), cudaMemcpyDeviceToHost, st));
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    K3_CUDA_TRY(cudaMemsetAsync(flag, 0, sizeof(int), st));
    if (bad) return K3MOE_ERR_BAD_SCALE;

    h->w_router = w->w_router;
    h->bias = w->select_bias;
    h->w_down = w->w_down;
    h->w_up = w->w_up;
    h->gamma = w->norm_gamma;
    for (int i = 0; i < 6; ++i) h->shared[i] = sh[i];
    h->aligned16 = al;
    if (al) {
        int rc = k3_tc_prepare(h, tabs, st);
        if (rc) return rc;
    }
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    h->loaded = true;
    return K3MOE_OK;
}

int k3moe_path_for(const k3moe_handle *h, int T)
{
    (void)T;
    if (!h) return K3MOE_ERR_ARG;
    if (h->cfg.path == K3MOE_PATH_GENERIC || !h->aligned16 || !k3_tc_available()) return K3MOE_PATH_GENERIC;
    return K3MOE_PATH_TENSOR;
}

size_t k3moe_workspace_bytes(const k3moe_handle *h, int T)
{
    if (!h || T < 0 || T > K3_MAX_TOKENS) return 0;
    k3_ws ws;
    k3_ws_layout(h, T, nullptr, &ws);
    return ws.bytes;
}

}  // extern "C"

int k3_ws_layout(const k3moe_handle *h, int T, void *base, k3_ws *ws)
{
    const k3moe_config &c = h->cfg;
    const size_t R = (size_t)T * c.top_k;
    const size_t Tn = T > 0 ? T : 1;
    Carver cv{(uint8_t *)base};
    ws->logits = cv.take<float>(Tn * c.n_experts);
    ws->h = cv.take<uint16_t>(Tn * c.latent);
    ws->idx = cv.take<int32_t>(R + 1);
    ws->wts = cv.take<float>(R + 1);
    ws->counts = cv.take<int32_t>(c.n_experts);
    ws->offsets = cv.take<int32_t>(c.n_experts + 1);
    ws->tok_of = cv.take<int32_t>(R + 1);
    ws->row_of = cv.take<int32_t>(R + 1);
    ws->meta = cv.take<int32_t>(16);
    ws->active = cv.take<int32_t>(c.n_experts);
    ws->tiles = cv.take<int32_t>(4 * (R + c.n_experts + 1));
    ws->gv_sync = cv.take<int32_t>(2 + R + c.n_experts);
    ws->act = cv.take<float>(R * c.inter + 1);          // fp32 (generic) or f16 (tensor)
    ws->y = cv.take<float>(R * c.latent + 1);
    // Tensor-path expert inputs in expert order: f16 h [R, L] (decode GEMV and tcgen05
    // tiles), with A8 through the GEMV later the MXFP8-rounded GLU output [R, I] as f16;
    // block-scaled A8 tiles: MXFP8 h [R, L] and GLU output [R, I], one byte each.  Before
    // the weights are loaded the tensor path is assumed (the generic path does not use it).
    {
        const size_t LI = (size_t)(c.latent > c.inter ? c.latent : c.inter);
        const bool gemv = R <= (size_t)c.n_experts * 24;
        const bool tensor = h->loaded ? k3moe_path_for(h, T) == K3MOE_PATH_TENSOR : c.path != K3MOE_PATH_GENERIC;
        size_t halves = 1;
        if (tensor && c.a8 && gemv) halves = R * LI;
        else if (tensor && c.a8) halves = (R * (size_t)(c.latent + c.inter) + 1) / 2;
        else if (tensor) halves = R * (size_t)c.latent;
        ws->hperm = cv.take<uint16_t>(halves + 1);
    }
    ws->hscale = cv.take<float>(R + 1);
    ws->ascale = cv.take<float>(R + 1);
    ws->nrm = cv.take<uint16_t>(Tn * c.latent);
    ws->o32 = cv.take<float>(Tn * c.hidden);
    {   // split-K partials for the decode-size dense GEMMs: up to K3_DENSE_MAX_SPLITS splits
        const size_t ep = (size_t)((c.n_experts + 15) & ~15);
        const size_t w = ep + c.latent > (size_t)c.hidden ? ep + c.latent : (size_t)c.hidden;
        ws->part_floats = T <= 256 ? (size_t)K3_DENSE_MAX_SPLITS * Tn * w : 1;
        ws->part = cv.take<float>(ws->part_floats);
    }
    ws->sact = cv.take<float>(c.shared_inter ? Tn * c.shared_inter : 1);
    ws->xs = cv.take<uint16_t>(c.shared_inter ? Tn * c.hidden : 1);
    ws->xscale = cv.take<float>(Tn);
    ws->xascale = cv.take<float>(Tn);
    ws->stage_x = cv.take<uint16_t>(Tn * c.hidden);
    ws->stage_out = cv.take<uint16_t>(Tn * c.hidden);
    ws->stage_idx = cv.take<int32_t>(R + 1);
    ws->stage_w = cv.take<float>(R + 1);
    ws->chunk_cnt = cv.take<int32_t>(T >= K3_PERM_CHUNKED_T
                                         ? (size_t)c.n_experts * ((T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK)
                                         : 1);
    ws->mxs = cv.take<uint8_t>(c.a8 ? R * (size_t)(c.latent + c.inter) / 32 + 16 : 1);
    ws->bytes = align_up(cv.off, 256);
    return K3MOE_OK;
}

static int forward_generic(k3moe_handle *h, const void *x, int T, void *out, const k3_ws &ws,
                           cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int H = c.hidden, L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int R = T * K;
    int rc;
    {   // router logits (fp32)
        k3_stage sg(h, K3MOE_STAGE_ROUTER, st);
        if ((rc = k3_launch_rows_gemm(x, 1, T, H, h->w_router, c.router_dtype == K3MOE_ROUTER_BF16, E,
                                      ws.logits, nullptr, 0, st)))
            return rc;
    }
    {   // latent h (BF16)
        k3_stage sg(h, K3MOE_STAGE_DOWN, st);
        if ((rc = k3_launch_rows_gemm(x, 1, T, H, h->w_down, 1, L, nullptr, ws.h, 0, st))) return rc;
        // A8: the routed experts read h as MXFP8
        if (c.a8 && (rc = k3_launch_mx8_rows(ws.h, 0, ws.h, 0, (size_t)T * L, h->d_status, h->num_sms, st)))
            return rc;
    }
    if ((rc = k3_launch_route(h, ws, T, 0, st))) return rc;   // top-K and the permutation
    {
        k3_stage sg(h, K3MOE_STAGE_GATE_UP, st);
        if ((rc = k3_launch_glu_generic(k3_act_of(h->cfg), ws.h, L, ws.tok_of, R, h->d_eptr[0], h->d_eptr[1], h->d_eptr[2],
                                        h->d_eptr[3], ws.offsets, E, I, (float *)ws.act, h->d_status,
                                        st)))
            return rc;
        // A8: the down projection reads the GLU output as MXFP8
        if (c.a8 && (rc = k3_launch_mx8_rows(ws.act, 1, ws.act, 1, (size_t)R * I, h->d_status, h->num_sms, st)))
            return rc;
    }
    {
        k3_stage sg(h, K3MOE_STAGE_EXPERT_DOWN, st);
        if ((rc = k3_launch_down_generic((const float *)ws.act, I, R, h->d_eptr[4], h->d_eptr[5],
                                         ws.offsets, E, L, (float *)ws.y, 0, st)))
            return rc;
    }
    {
        k3_stage sg(h, K3MOE_STAGE_COMBINE, st);
        if ((rc = k3_launch_combine_norm(ws.y, 0, ws.row_of, ws.wts, h->gamma, T, K, L, c.rms_eps,
                                         ws.nrm, st)))
            return rc;
    }
    {
        k3_stage sg(h, K3MOE_STAGE_UP, st);
        if ((rc = k3_launch_rows_gemm(ws.nrm, 1, T, L, h->w_up, 1, H, ws.o32, nullptr, 0, st)))
            return rc;
    }
    if (c.shared_inter > 0) {
        k3_stage sg(h, K3MOE_STAGE_SHARED, st);
        const int S = c.shared_inter;
        if ((rc = k3_launch_glu_generic(k3_act_of(h->cfg), (const uint16_t *)x, H, nullptr, T, k3_shared_tab(h, 0),
                                        k3_shared_tab(h, 1), k3_shared_tab(h, 2), k3_shared_tab(h, 3),
                                        nullptr, 1, S, (float *)ws.sact, h->d_status, st)))
            return rc;
        if ((rc = k3_launch_down_generic((const float *)ws.sact, S, T, k3_shared_tab(h, 4),
                                         k3_shared_tab(h, 5), nullptr, 1, H, ws.o32, 1, st)))
            return rc;
    }
    k3_stage sg(h, K3MOE_STAGE_FINISH, st);
    return k3_launch_finish(ws.o32, T * H, (uint16_t *)out, st);
}

extern "C" {

static int forward_impl(k3moe_handle *h, const void *x, int T, void *out, int32_t *idx_out,
                        float *w_out, void *workspace, size_t workspace_bytes, cudaStream_t st,
                        bool staged)
{
    if (!h) return K3MOE_ERR_ARG;
    if (!h->loaded) return K3MOE_ERR_STATE;
    if (T < 0 || T > K3_MAX_TOKENS) return K3MOE_ERR_ARG;
    if (T == 0) return K3MOE_OK;
    if (!x || !out || !workspace) return K3MOE_ERR_ARG;
    const k3moe_config &c = h->cfg;
    if ((uintptr_t)x % 16 || (uintptr_t)out % 16) return K3MOE_ERR_ALIGN;
    if ((uintptr_t)workspace % 256) return K3MOE_ERR_ALIGN;
    const size_t xb = (size_t)T * c.hidden * 2;
    if (overlaps(x, xb, out, xb)) return K3MOE_ERR_ALIAS;
    if (idx_out && overlaps(x, xb, idx_out, (size_t)T * c.top_k * 4)) return K3MOE_ERR_ALIAS;
    if (w_out && overlaps(x, xb, w_out, (size_t)T * c.top_k * 4)) return K3MOE_ERR_ALIAS;
    k3_ws ws;
    k3_ws_layout(h, T, workspace, &ws);
    if (workspace_bytes < ws.bytes) return K3MOE_ERR_WORKSPACE;
    // the compute part of the workspace ends where the host-call staging begins
    const size_t compute_bytes = (size_t)((uint8_t *)ws.stage_x - (uint8_t *)workspace);
    if (!staged && (overlaps(workspace, ws.bytes, x, xb) || overlaps(workspace, ws.bytes, out, xb)))
        return K3MOE_ERR_ALIAS;
    if (staged && (overlaps(workspace, compute_bytes, x, xb) || overlaps(workspace, compute_bytes, out, xb)))
        return K3MOE_ERR_ALIAS;
    int dev = 0;
    K3_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != h->device) return K3MOE_ERR_STATE;
    int rc = (k3moe_path_for(h, T) == K3MOE_PATH_TENSOR) ? k3_forward_tc(h, x, T, out, ws, st)
                                                         : forward_generic(h, x, T, out, ws, st);
    if (h->prof && h->prof->on && h->prof->pos < k3_prof::RING) h->prof->pos++;
    if (rc) return rc;
    const size_t kb = (size_t)T * c.top_k * 4;
    if (idx_out) K3_CUDA_TRY(cudaMemcpyAsync(idx_out, ws.idx, kb, cudaMemcpyDeviceToDevice, st));
    if (w_out) K3_CUDA_TRY(cudaMemcpyAsync(w_out, ws.wts, kb, cudaMemcpyDeviceToDevice, st));
    return K3MOE_OK;
}

int k3moe_forward(k3moe_handle *h, const void *x, int T, void *out, int32_t *idx_out, float *w_out,
                  void *workspace, size_t workspace_bytes, cudaStream_t st)
{
    return forward_impl(h, x, T, out, idx_out, w_out, workspace, workspace_bytes, st, false);
}

int k3moe_forward_host(k3moe_handle *h, const void *x_host, int T, void *out_host, int32_t *idx_host,
                       float *w_host, void *workspace, size_t workspace_bytes, cudaStream_t st)
{
    if (!h) return K3MOE_ERR_ARG;
    if (!h->loaded) return K3MOE_ERR_STATE;
    if (T < 0 || T > K3_MAX_TOKENS) return K3MOE_ERR_ARG;
    if (T == 0) return K3MOE_OK;
    if (!x_host || !out_host || !workspace) return K3MOE_ERR_ARG;
    if ((uintptr_t)workspace % 256) return K3MOE_ERR_ALIGN;
    const k3moe_config &c = h->cfg;
    k3_ws ws;
    k3_ws_layout(h, T, workspace, &ws);
    if (workspace_bytes < ws.bytes) return K3MOE_ERR_WORKSPACE;
    const size_t xb = (size_t)T * c.hidden * 2, kb = (size_t)T * c.top_k * 4;
    K3_CUDA_TRY(cudaMemcpyAsync(ws.stage_x, x_host, xb, cudaMemcpyHostToDevice, st));
    int rc = forward_impl(h, ws.stage_x, T, ws.stage_out, idx_host ? ws.stage_idx : nullptr,
                          w_host ? ws.stage_w : nullptr, workspace, workspace_bytes, st, true);
    if (rc) return rc;
    K3_CUDA_TRY(cudaMemcpyAsync(out_host, ws.stage_out, xb, cudaMemcpyDeviceToHost, st));
    if (idx_host) K3_CUDA_TRY(cudaMemcpyAsync(idx_host, ws.stage_idx, kb, cudaMemcpyDeviceToHost, st));
    if (w_host) K3_CUDA_TRY(cudaMemcpyAsync(w_host, ws.stage_w, kb, cudaMemcpyDeviceToHost, st));
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    return K3MOE_OK;
}

int k3moe_status(k3moe_handle *h, cudaStream_t st)
{
    if (!h || !h->loaded) return K3MOE_ERR_STATE;
    int v[ST_COUNT] = {0};
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    K3_CUDA_TRY(cudaMemcpy(v, h->d_status, sizeof(v), cudaMemcpyDeviceToHost));
    K3_CUDA_TRY(cudaMemsetAsync(h->d_status, 0, sizeof(int) * 2, st));
    // a device-side failure may have stopped a dense GEMM between its tiles' arrivals:
    // its split-K counters start from zero again
    if (v[ST_CODE]) K3_CUDA_TRY(cudaMemsetAsync(h->d_dense_cnt, 0, sizeof(int) * h->dense_cnt_n, st));
    K3_CUDA_TRY(cudaStreamSynchronize(st));
    return v[ST_CODE];
}

int k3moe_debug_dequant(const uint8_t *packed, const uint8_t *scale, int rows, int cols, float *out,
                        cudaStream_t st)
{
    if (!packed || !scale || !out || rows < 0 || cols < 0) return K3MOE_ERR_ARG;
    if (cols % 32) return K3MOE_ERR_SHAPE;
    return k3_launch_dequant_debug(packed, scale, rows, cols, out, st);
}

int k3moe_debug_wait_timeout(k3moe_handle *h, int spin_limit, cudaStream_t st)
{
    if (!h || !h->loaded) return K3MOE_ERR_STATE;
    if (spin_limit < 1) return K3MOE_ERR_ARG;
    return k3_launch_wait_debug(h->d_status, spin_limit, st);
}

}  // extern "C"

extern "C" size_t k3moe_qb_workspace_bytes(const k3moe_handle *h, int T, int nbins)
{
    if (!h || T < 2 || nbins < 1 || nbins > 8192) return 0;
    return k3_qb_workspace_bytes(T, h->cfg.n_experts, nbins);
}

extern "C" int k3moe_qb_bias(k3moe_handle *h, const float *logits, int T, const float *bias_in, float *bias_out,
                             int nbins, void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (!h || !logits || !bias_out || !workspace) return K3MOE_ERR_ARG;
    if (T < 2 || nbins < 1 || nbins > 8192) return K3MOE_ERR_ARG;
    if (h->cfg.top_k + 1 > h->cfg.n_experts) return K3MOE_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (dev != h->device) return K3MOE_ERR_STATE;
    return k3_qb_bias(h, logits, T, bias_in, bias_out, nbins, workspace, workspace_bytes, stream);
}

static int ep_check(const k3moe_handle *h, int n_ranks, int S)
{
    if (!h) return K3MOE_ERR_ARG;
    if (!h->loaded) return K3MOE_ERR_STATE;
    const int E = h->cfg.n_experts, K = h->cfg.top_k;
    if (E > 1024 || K > 32) return K3MOE_ERR_UNSUPPORTED;
    if (n_ranks < 1 || n_ranks > E || E % n_ranks || S < 1) return K3MOE_ERR_ARG;
    if ((long long)n_ranks * S * K >= (1LL << 31)) return K3MOE_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (dev != h->device) return K3MOE_ERR_STATE;
    return K3MOE_OK;
}

static bool ep_plan_ok(const k3moe_ep_plan *p)
{
    return p && p->seg && p->rank_seg && p->exp_off && p->exp_seg && p->info;
}

extern "C" int k3moe_ep_plan_compute(k3moe_handle *h, const int32_t *counts, int n_ranks, int tokens_per_rank,
                                     const k3moe_ep_plan *plan, cudaStream_t stream)
{
    if (!counts || !ep_plan_ok(plan)) return K3MOE_ERR_ARG;
    const int rc = ep_check(h, n_ranks, tokens_per_rank);
    if (rc) return rc;
    return k3_ep_plan(h, counts, n_ranks, tokens_per_rank * h->cfg.top_k, plan, stream);
}

extern "C" size_t k3moe_ep_dispatch_workspace_bytes(const k3moe_handle *h, int tokens_per_rank)
{
    if (!h || tokens_per_rank < 1 || (long long)tokens_per_rank * h->cfg.top_k >= (1LL << 31)) return 0;
    return k3_ep_dispatch_workspace_bytes(tokens_per_rank, h->cfg.n_experts);
}

extern "C" int k3moe_ep_dispatch(k3moe_handle *h, const int32_t *idx, int tokens_per_rank, int src_rank,
                                 const int32_t *counts, int n_ranks, const k3moe_ep_plan *plan, int32_t *dest_rank,
                                 int32_t *dest_row, void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (!idx || !counts || !dest_rank || !dest_row || !ep_plan_ok(plan)) return K3MOE_ERR_ARG;
    const int rc = ep_check(h, n_ranks, tokens_per_rank);
    if (rc) return rc;
    if (src_rank < 0 || src_rank >= n_ranks) return K3MOE_ERR_ARG;
    if (!workspace || workspace_bytes < k3_ep_dispatch_workspace_bytes(tokens_per_rank, h->cfg.n_experts))
        return K3MOE_ERR_WORKSPACE;
    return k3_ep_dispatch(h, idx, tokens_per_rank, src_rank, counts, n_ranks, plan, dest_rank, dest_row, workspace,
                          stream);
}
