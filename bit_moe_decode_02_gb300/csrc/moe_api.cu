// moe_api.cu -- the C ABI declared in include/moe.h: handle, argument checks,
// resident weight arena, workspace and the launches of the layer kernels.
//
// All tables the kernels need are fixed at moe_create / moe_load_experts; a
// forward call does no host-side work that depends on the routing (the pages'
// lesson: per-token host setup once cost 10.65 ms of a 36.95 ms token,
// "Amortizing the per-token host-sync setup tax ...", section 3), and it
// allocates nothing (the grow-only buffer cache that reallocated on every
// count change, TinyTitan tracker D114).
//
// Resident layout, per layer: [gate_up of E experts][down of E experts]
// [gate_up biases bf16 [E][2I]][down biases bf16 [E][H]], 256-byte aligned.
// MXFP4 experts are in the 128-row tile layout of the tensor-core kernels,
// int4 experts in the 64-row unit layout of the int4 kernel (each described
// with its kernel); both hold exactly the caller's bytes, reordered.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

int moe::set_error(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

struct moe_handle {
    moe_config cfg{};
    int device = 0;
    int num_sms = 0;
    bool mxfp4 = false;
    // caller-layout tensor sizes in bytes (one layer, all experts)
    size_t gu_codes_b = 0, gu_scales_b = 0, gu_bias_b = 0;
    size_t dn_codes_b = 0, dn_scales_b = 0, dn_bias_b = 0;
    // resident layout
    size_t gu_expert = 0, dn_expert = 0;      // bytes of one expert's projection
    size_t off_dn = 0, off_gu_bias = 0, off_dn_bias = 0, layer_stride = 0;
    uint8_t* arena = nullptr;
    std::vector<char> loaded;
    // decode workspace (both formats): per-CTA output copies and the counters
    size_t dec_smem = 0;                      // dynamic shared memory of the decode kernel
    float* part = nullptr;                    // [G][H][4]
    unsigned long long* cnt = nullptr;        // xcnt, done (only grow)
    // MXFP4 decode: split-unit partials and flags, the layer's x terms
    float* gpart = nullptr;
    unsigned* pflag = nullptr;
    uint8_t* xt = nullptr;
    // batched path (MXFP4, M > 4)
    bool batched = false;
    int max_tiles = 0;
    int* b_int = nullptr;                     // idx | slot | etile | erow | ntiles
    float* b_wt = nullptr;
    moe::TokTile* b_tiles = nullptr;
    uint8_t* b_xq = nullptr;
    uint8_t* b_xsf = nullptr;
    uint8_t* b_hq = nullptr;
    uint8_t* b_hsf = nullptr;
    float* b_y = nullptr;
    int b_f16 = 0;                            // batched numerics: 0 MXFP4 activations, 1 bf16
    uint8_t* b_a16 = nullptr;                 // bf16 variant: x tiles, then h tiles (allocated on selection)
    int last_bM = 0, last_bk = 0;             // M and top_k of the last batched call
    // in-kernel router: per layer W bf16 [E][H] then the bias bf16 [E]
    // (rw_stride bytes a layer; allocated by the first moe_load_router), and
    // the logits of the last call [max(max_tokens, 4)][E]
    uint8_t* rw = nullptr;
    size_t rw_stride = 0;
    std::vector<char> rloaded;
    float* rlog = nullptr;
    int* stats = nullptr;                     // distinct experts of the last call on each layer
    int* status = nullptr;
    // staging for moe_forward_host: [x][residual / out][logits] in pinned host
    // memory mapped into the device's address space (st_dev is its device
    // address): the layer kernel reads the call's inputs from it and writes the
    // result into it directly, over the host-device link
    uint8_t* st_dev = nullptr;
    uint8_t* st_host = nullptr;
    size_t st_off_r = 0, st_off_l = 0, st_bytes = 0;
    // cross-CTA waits of the decode kernels (moe_debug_set_wait)
    int spin_limit = moe::kSpinLimit;
    int skip_cta = -1;
    float sw_alpha = 1.0f, sw_limit = INFINITY, sw_beta = 0.0f;   // the SwiGLU form (moe_set_swiglu)
    int last_steps = 0;        // layer calls of the last forward call: layers
    int last_first_layer = 0;  // last_first_layer, + 1, ... (mod L)
    int last_launches = 0;
};

namespace {

int check_cfg(const moe_config* c)
{
    if (!c)
        return fail(MOE_ERR_INVALID_ARG, "moe_create: cfg is NULL");
    if (c->hidden <= 0 || c->hidden % 64 || c->hidden > moe::kMaxK)
        return fail(MOE_ERR_INVALID_ARG, "hidden=%d must be a positive multiple of 64, <= %d",
                    c->hidden, moe::kMaxK);
    if (c->intermediate <= 0 || c->intermediate % 64 || c->intermediate > moe::kMaxK)
        return fail(MOE_ERR_INVALID_ARG, "intermediate=%d must be a positive multiple of 64, <= %d",
                    c->intermediate, moe::kMaxK);
    if (c->num_experts < 1 || c->num_experts > moe::kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "num_experts=%d must be in 1..%d", c->num_experts,
                    moe::kMaxExperts);
    if (c->num_layers < 1)
        return fail(MOE_ERR_INVALID_ARG, "num_layers=%d must be >= 1", c->num_layers);
    if (c->max_tokens < 1 || c->max_tokens > moe::kMaxBatchTokens)
        return fail(MOE_ERR_INVALID_ARG, "max_tokens=%d must be in 1..%d", c->max_tokens,
                    moe::kMaxBatchTokens);
    if (c->max_top_k < 1 || c->max_top_k > moe::kMaxTopK || c->max_top_k > c->num_experts)
        return fail(MOE_ERR_INVALID_ARG, "max_top_k=%d must be in 1..min(num_experts, %d)",
                    c->max_top_k, moe::kMaxTopK);
    if (c->format == MOE_FMT_MXFP4) {
        if (c->group != 32)
            return fail(MOE_ERR_INVALID_ARG, "MXFP4 needs group == 32 (got %d)", c->group);
    } else if (c->format == MOE_FMT_INT4) {
        if (c->group < 32 || c->group % 32 || c->hidden % c->group || c->intermediate % c->group)
            return fail(MOE_ERR_INVALID_ARG,
                        "int4 group=%d must be a multiple of 32 dividing hidden and intermediate",
                        c->group);
    } else {
        return fail(MOE_ERR_INVALID_ARG, "format=%d is neither MOE_FMT_MXFP4 nor MOE_FMT_INT4",
                    c->format);
    }
    if (c->has_bias != 0 && c->has_bias != 1)
        return fail(MOE_ERR_INVALID_ARG, "has_bias must be 0 or 1");
    if (c->max_tokens > moe::kMaxTokens && c->format != MOE_FMT_MXFP4)
        return fail(MOE_ERR_UNSUPPORTED, "max_tokens=%d > %d (the tensor-core batched path) needs "
                    "MOE_FMT_MXFP4", c->max_tokens, moe::kMaxTokens);
    return MOE_OK;
}

void free_handle(moe_handle* h)
{
    if (!h)
        return;
    cudaFree(h->arena);
    cudaFree(h->part);
    cudaFree(h->cnt);
    cudaFree(h->gpart);
    cudaFree(h->pflag);
    cudaFree(h->xt);
    cudaFree(h->b_int);
    cudaFree(h->b_wt);
    cudaFree(h->b_tiles);
    cudaFree(h->b_xq);
    cudaFree(h->b_xsf);
    cudaFree(h->b_hq);
    cudaFree(h->b_hsf);
    cudaFree(h->b_y);
    cudaFree(h->b_a16);
    cudaFree(h->stats);
    cudaFree(h->status);
    cudaFree(h->rw);
    cudaFree(h->rlog);
    cudaFreeHost(h->st_host);
    delete h;
}

template <typename T>
int dev_alloc(T** p, size_t bytes, const char* what)
{
    cudaError_t e = cudaMalloc((void**)p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return fail(MOE_ERR_OOM, "cudaMalloc(%zu bytes) for %s failed: %s", bytes, what,
                    cudaGetErrorString(e));
    }
    return MOE_OK;
}

const uint16_t* bias0(const moe_handle* h, size_t off)
{
    return h->cfg.has_bias ? reinterpret_cast<const uint16_t*>(h->arena + off) : nullptr;
}

// Parameters of the MXFP4 decode kernel for `ncalls` calls from `layer0`
// (the caller sets the inputs, outputs and strides).
moe::DecodeTcParams tc_params(const moe_handle* h, int layer0, int ncalls)
{
    const moe_config& c = h->cfg;
    moe::DecodeTcParams p{};
    p.resid_every = 1;
    p.sw_alpha = h->sw_alpha;
    p.sw_limit = h->sw_limit;
    p.sw_beta = h->sw_beta;
    p.gu = h->arena;
    p.dn = h->arena + h->off_dn;
    p.layer_stride = (long long)h->layer_stride;
    p.gu_expert = (long long)h->gu_expert;
    p.dn_expert = (long long)h->dn_expert;
    p.gu_bias = bias0(h, h->off_gu_bias);
    p.dn_bias = bias0(h, h->off_dn_bias);
    p.bias_stride = (long long)h->layer_stride;
    p.ncalls = ncalls;
    p.layer0 = layer0;
    p.nlayers = c.num_layers;
    p.part = h->part;
    p.gpart = h->gpart;
    p.pflag = h->pflag;
    p.xt = h->xt;
    p.xcnt = h->cnt;
    p.done = h->cnt + 1;
    p.status = h->status;
    p.nu_out = h->stats;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.smem_bytes = (int)h->dec_smem;
    p.spin_limit = h->spin_limit;
    p.skip_cta = h->skip_cta;
    return p;
}

moe::DecodeI4Params i4_params(const moe_handle* h, int layer0, int ncalls)
{
    const moe_config& c = h->cfg;
    moe::DecodeI4Params p{};
    p.resid_every = 1;
    p.sw_alpha = h->sw_alpha;
    p.sw_limit = h->sw_limit;
    p.sw_beta = h->sw_beta;
    p.gu = h->arena;
    p.dn = h->arena + h->off_dn;
    p.layer_stride = (long long)h->layer_stride;
    p.gu_expert = (long long)h->gu_expert;
    p.dn_expert = (long long)h->dn_expert;
    p.gu_bias = bias0(h, h->off_gu_bias);
    p.dn_bias = bias0(h, h->off_dn_bias);
    p.bias_stride = (long long)h->layer_stride;
    p.ncalls = ncalls;
    p.layer0 = layer0;
    p.nlayers = c.num_layers;
    p.part = h->part;
    p.done = h->cnt + 1;
    p.status = h->status;
    p.nu_out = h->stats;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.group = c.group;
    p.smem_bytes = (int)h->dec_smem;
    p.spin_limit = h->spin_limit;
    p.skip_cta = h->skip_cta;
    return p;
}

// A sequence of `n` decode calls in one launch: call s runs layer (layer0 + s)
// mod L on logits + s * ls, x + s * xs (x may be NULL: the normalised
// residual), resid + s * rs and out_f32 + s * fs (bytes).
cudaError_t launch_seq(const moe_handle* h, int layer0, int n, const float* logits, long long ls, const void* x,
                       long long xs, void* resid, long long rs, float* out_f32, long long fs, int M, int k,
                       cudaStream_t s, int resid_every = 1)
{
    if (h->mxfp4) {
        moe::DecodeTcParams p = tc_params(h, layer0, n);
        p.logits = logits;
        p.router = logits ? nullptr : reinterpret_cast<const uint16_t*>(h->rw);
        p.router_stride = (long long)h->rw_stride;
        p.rlog = h->rlog;
        p.logits_stride = ls;
        p.x = static_cast<const uint16_t*>(x);
        p.x_stride = xs;
        p.resid = static_cast<uint16_t*>(resid);
        p.resid_stride = rs;
        p.resid_every = resid_every;
        p.out_f32 = out_f32;
        p.out_f32_stride = fs;
        p.M = M;
        p.k = k;
        return moe::launch_decode_tc(p, h->dec_smem, h->num_sms, s);
    }
    moe::DecodeI4Params p = i4_params(h, layer0, n);
    p.logits = logits;
    p.router = logits ? nullptr : reinterpret_cast<const uint16_t*>(h->rw);
    p.router_stride = (long long)h->rw_stride;
    p.rlog = h->rlog;
    p.logits_stride = ls;
    p.x = static_cast<const uint16_t*>(x);
    p.x_stride = xs;
    p.resid = static_cast<uint16_t*>(resid);
    p.resid_stride = rs;
    p.resid_every = resid_every;
    p.out_f32 = out_f32;
    p.out_f32_stride = fs;
    p.M = M;
    p.k = k;
    return moe::launch_decode_i4(p, h->dec_smem, h->num_sms, s);
}

// One decode layer call.
cudaError_t launch_decode(const moe_handle* h, int layer, const float* logits, const void* x, void* resid, int M,
                          int k, cudaStream_t s, float* out_f32 = nullptr)
{
    return launch_seq(h, layer, 1, logits, 0, x, 0, resid, 0, out_f32, 0, M, k, s);
}

// Decode workspace and kernel set-up (both formats).
int create_decode(moe_handle* h)
{
    const moe_config& c = h->cfg;
    const int H = c.hidden, G = h->num_sms;
    int rc;
    if ((rc = dev_alloc(&h->part, moe::tc_part_bytes(G, H), "per-CTA outputs")) ||
        (rc = dev_alloc(&h->cnt, moe::kTcCounterWords * sizeof(unsigned long long), "counters")))
        return rc;
    cudaError_t e = cudaMemset(h->cnt, 0, moe::kTcCounterWords * sizeof(unsigned long long));
    if (e != cudaSuccess)
        return cuda_fail(e, "counters");
    int dev = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return cuda_fail(e, "shared memory limit");
    if (h->mxfp4) {
        if ((rc = dev_alloc(&h->gpart, (size_t)G * moe::kRowTile * 4 * sizeof(float), "split-unit partials")) ||
            (rc = dev_alloc(&h->pflag, (size_t)G * sizeof(unsigned), "split-unit flags")) ||
            (rc = dev_alloc(&h->xt, moe::tc_terms_bytes(H), "x terms")))
            return rc;
        // x-term rows past M * 8 are never written and feed MMA columns nobody reads:
        // keep them zero (valid E2M1 codes, E8M0 byte 0) instead of leftover bytes
        if ((e = cudaMemset(h->xt, 0, moe::tc_terms_bytes(H))) != cudaSuccess ||
            (e = cudaMemset(h->pflag, 0, (size_t)G * sizeof(unsigned))) != cudaSuccess)
            return cuda_fail(e, "decode workspace");
        h->dec_smem = (size_t)optin - moe::decode_tc_static_smem();
        if ((e = moe::prepare_decode_tc(h->dec_smem)) != cudaSuccess)
            return cuda_fail(e, "tensor-core decode kernel set-up");
    } else {
        h->dec_smem = (size_t)optin - moe::decode_i4_static_smem();
        // the int4 kernel's tail (x as f16, sums, h', the output copy) and at least two stages
        const size_t tail = (size_t)4 * (H + 8) * 2 + 2 * 128 * 16 + 2 * 4 * 64 * 2 + (size_t)H * 16 + 128;
        if (h->dec_smem < tail + 2 * (size_t)moe::kI4Slot)
            return fail(MOE_ERR_UNSUPPORTED, "hidden=%d leaves no room for the int4 kernel's stage ring", H);
        if ((e = moe::prepare_decode_i4(h->dec_smem)) != cudaSuccess)
            return cuda_fail(e, "int4 decode kernel set-up");
    }
    return MOE_OK;
}

// Workspace of the batched path.
int create_batched(moe_handle* h)
{
    const moe_config& c = h->cfg;
    const int H = c.hidden, I = c.intermediate, E = c.num_experts;
    const size_t Mk = (size_t)c.max_tokens * c.max_top_k;
    h->batched = true;
    h->max_tiles = moe::max_tok_tiles((int)Mk, E);
    const size_t rows = Mk + 16 * (size_t)h->max_tiles;   // padded activation rows, upper bound
    int rc;
    if ((rc = dev_alloc(&h->b_int, (4 * Mk + 1) * sizeof(int), "batched tables")) ||
        (rc = dev_alloc(&h->b_wt, Mk * sizeof(float), "routing weights")) ||
        (rc = dev_alloc(&h->b_tiles, h->max_tiles * sizeof(moe::TokTile), "token tiles")) ||
        (rc = dev_alloc(&h->b_xq, rows * H / 2, "x codes")) ||
        (rc = dev_alloc(&h->b_xsf, (size_t)h->max_tiles * moe::ceil_div(H, 128) * moe::kSfChunk, "x scales")) ||
        (rc = dev_alloc(&h->b_hq, rows * I / 2, "h codes")) ||
        (rc = dev_alloc(&h->b_hsf, (size_t)h->max_tiles * moe::ceil_div(I, 128) * moe::kSfChunk, "h scales")) ||
        (rc = dev_alloc(&h->b_y, Mk * H * sizeof(float), "batched y")))
        return rc;
    cudaError_t e = moe::prepare_batched_kernels();
    if (e != cudaSuccess)
        return cuda_fail(e, "batched kernel set-up");
    return MOE_OK;
}

moe::BatchParams batch_params(const moe_handle* h, int layer)
{
    const moe_config& c = h->cfg;
    const size_t Mk = (size_t)c.max_tokens * c.max_top_k;
    const uint8_t* base = h->arena + (size_t)layer * h->layer_stride;
    moe::BatchParams p{};
    p.gu = base;
    p.dn = base + h->off_dn;
    p.gu_expert = (long long)h->gu_expert;
    p.dn_expert = (long long)h->dn_expert;
    p.gu_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(base + h->off_gu_bias) : nullptr;
    p.dn_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(base + h->off_dn_bias) : nullptr;
    p.idx = h->b_int;
    p.slot = h->b_int + Mk;
    p.etile = h->b_int + 2 * Mk;
    p.erow = h->b_int + 3 * Mk;
    p.ntiles = h->b_int + 4 * Mk;
    p.wt = h->b_wt;
    p.tiles = h->b_tiles;
    p.xq = h->b_xq;
    p.xsf = h->b_xsf;
    p.hq = h->b_hq;
    p.hsf = h->b_hsf;
    p.y = h->b_y;
    if (h->b_f16) {
        const size_t rows = Mk + 16 * (size_t)h->max_tiles;
        p.f16 = 1;
        p.x16 = h->b_a16;
        p.h16 = h->b_a16 + rows * c.hidden * 2;
    }
    p.status = h->status;
    p.nu_out = h->stats + layer;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.max_tiles = h->max_tiles;
    p.sw_alpha = h->sw_alpha;
    p.sw_limit = h->sw_limit;
    p.sw_beta = h->sw_beta;
    return p;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

int check_forward_args(const moe_handle* h, int M, int top_k)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
    if (M < 1 || M > h->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "M=%d must be in 1..max_tokens=%d", M, h->cfg.max_tokens);
    if (top_k < 1 || top_k > h->cfg.max_top_k)
        return fail(MOE_ERR_INVALID_ARG, "top_k=%d must be in 1..max_top_k=%d", top_k,
                    h->cfg.max_top_k);
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// False only for host memory the device cannot read at the same address
// (pageable, or page-locked but not mapped there).  A query that fails (for
// instance inside a stream capture that forbids it) proves nothing and passes.
bool device_accessible(const void* p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return true;
    }
    if (a.type == cudaMemoryTypeUnregistered)
        return false;
    return a.type != cudaMemoryTypeHost || a.devicePointer == p;
}

// Router weights for the layers (layer0 + s) mod L, s < n, when the logits are
// to be computed in the kernel (the caller passed none).
int check_router(const moe_handle* h, int layer0, int n, const char* who)
{
    const int L = h->cfg.num_layers;
    for (int s = 0; s < n && s < L; ++s)
        if (!h->rloaded[(layer0 + s) % L])
            return fail(MOE_ERR_NOT_LOADED, "%s: no router logits given and layer %d has no router weights "
                        "(moe_load_router)", who, (layer0 + s) % L);
    return MOE_OK;
}

int check_all_loaded(const moe_handle* h, const char* who)
{
    for (int l = 0; l < h->cfg.num_layers; ++l)
        if (!h->loaded[l])
            return fail(MOE_ERR_NOT_LOADED, "%s: layer %d has no experts loaded", who, l);
    return MOE_OK;
}

int forward_impl(moe_handle* h, int layer, const void* x_bf16, const float* router_logits, int M,
                 int top_k, void* out_bf16, float* out_f32, void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!x_bf16 || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x and out must not be NULL");
    if (!aligned16(x_bf16) || !aligned16(out_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x, logits and out must be 16-byte aligned");
    const size_t nb = (size_t)M * h->cfg.hidden * 2;
    if (overlaps(x_bf16, nb, out_bf16, nb))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x overlaps out");
    if (!h->loaded[layer])
        return fail(MOE_ERR_NOT_LOADED, "moe_forward: layer %d has no experts loaded", layer);
    if (!router_logits && (rc = check_router(h, layer, 1, "moe_forward")) != MOE_OK)
        return rc;
    if (M > moe::kMaxTokens) {
        moe::BatchParams b = batch_params(h, layer);
        if (!router_logits) {
            // the router GEMV first, into the handle's logits buffer
            cudaError_t e = moe::launch_router_gemv(static_cast<const uint16_t*>(x_bf16),
                                                    reinterpret_cast<const uint16_t*>(h->rw + layer * h->rw_stride),
                                                    M, h->cfg.hidden, h->cfg.num_experts, h->rlog,
                                                    (cudaStream_t)stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "moe_forward (router) launch");
            router_logits = h->rlog;
        }
        b.logits = router_logits;
        b.x = static_cast<const uint16_t*>(x_bf16);
        b.resid = static_cast<uint16_t*>(out_bf16);
        b.out_f32 = out_f32;
        b.M = M;
        b.k = top_k;
        int launches = 0;
        cudaError_t e = moe::launch_batched(b, h->num_sms, (cudaStream_t)stream, &launches);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_forward (batched) launch");
        h->last_steps = 1;
        h->last_first_layer = layer;
        h->last_launches = launches + (router_logits == h->rlog ? 1 : 0);
        h->last_bM = M;
        h->last_bk = top_k;
        return MOE_OK;
    }
    cudaError_t e = launch_decode(h, layer, router_logits, x_bf16, out_bf16, M, top_k, (cudaStream_t)stream,
                                  out_f32);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward launch");
    h->last_steps = 1;
    h->last_first_layer = layer;
    h->last_launches = 1;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err; }

int moe_create(const moe_config* cfg, moe_handle** out)
{
    if (!out)
        return fail(MOE_ERR_INVALID_ARG, "moe_create: out is NULL");
    *out = nullptr;
    int rc = check_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    moe_handle* h = new (std::nothrow) moe_handle();
    if (!h)
        return fail(MOE_ERR_OOM, "host allocation failed");
    h->cfg = *cfg;
    const moe_config& c = h->cfg;
    const size_t H = c.hidden, I = c.intermediate, E = c.num_experts;
    h->mxfp4 = c.format == MOE_FMT_MXFP4;
    const size_t sbh = h->mxfp4 ? H / 32 : 2 * H / c.group;
    const size_t sbi = h->mxfp4 ? I / 32 : 2 * I / c.group;
    h->gu_codes_b = E * 2 * I * H / 2;
    h->gu_scales_b = E * 2 * I * sbh;
    h->gu_bias_b = c.has_bias ? E * 2 * I * 2 : 0;
    h->dn_codes_b = E * H * I / 2;
    h->dn_scales_b = E * H * sbi;
    h->dn_bias_b = c.has_bias ? E * H * 2 : 0;
    if (h->mxfp4) {
        h->gu_expert = (size_t)moe::tile_proj_bytes(2 * (int)I, (int)H);   // interleaved gate_up
        h->dn_expert = (size_t)moe::tile_proj_bytes((int)H, (int)I);
    } else {
        h->gu_expert = (I / 64) * (size_t)moe::i4_unit_bytes((int)H, c.group, 0);
        h->dn_expert = (I / 64) * (size_t)moe::i4_unit_bytes((int)H, c.group, 1);
    }
    size_t off = align_up(E * h->gu_expert, 256);
    h->off_dn = off;
    off = align_up(off + E * h->dn_expert, 256);
    h->off_gu_bias = off;
    off = align_up(off + h->gu_bias_b, 256);
    h->off_dn_bias = off;
    h->layer_stride = align_up(off + h->dn_bias_b, 256);

    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "cudaGetDevice / SM count");
    }
    const size_t Mx = c.max_tokens;
    h->st_off_r = align_up(Mx * H * 2, 256);
    h->st_off_l = h->st_off_r + align_up(Mx * H * 2, 256);
    h->st_bytes = h->st_off_l + Mx * E * sizeof(float);
    if ((rc = dev_alloc(&h->arena, h->layer_stride * c.num_layers, "expert weights")) ||
        (rc = dev_alloc(&h->stats, c.num_layers * sizeof(int), "stats")) ||
        (rc = dev_alloc(&h->rlog, (size_t)std::max(c.max_tokens, moe::kMaxTokens) * E * sizeof(float),
                        "router logits")) ||
        (rc = dev_alloc(&h->status, sizeof(int), "status"))) {
        free_handle(h);
        return rc;
    }
    if ((e = cudaHostAlloc((void**)&h->st_host, h->st_bytes, cudaHostAllocMapped)) != cudaSuccess ||
        (e = cudaHostGetDevicePointer((void**)&h->st_dev, h->st_host, 0)) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return fail(MOE_ERR_OOM, "mapped pinned host staging (%zu bytes) failed: %s", h->st_bytes,
                    cudaGetErrorString(e));
    }
    if ((e = cudaMemset(h->stats, 0, c.num_layers * sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(h->status, 0, sizeof(int))) != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "moe_create setup");
    }
    if ((rc = create_decode(h)) != MOE_OK ||
        (c.max_tokens > moe::kMaxTokens && (rc = create_batched(h)) != MOE_OK)) {
        free_handle(h);
        return rc;
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "moe_create setup");
    }
    h->loaded.assign(c.num_layers, 0);
    h->rloaded.assign(c.num_layers, 0);
    *out = h;
    g_err[0] = 0;
    return MOE_OK;
}

void moe_destroy(moe_handle* h)
{
    if (!h)
        return;
    cudaDeviceSynchronize();
    free_handle(h);
}

long long moe_expert_bytes(const moe_handle* h)
{
    if (!h)
        return 0;
    const size_t E = h->cfg.num_experts;
    return (long long)((h->gu_codes_b + h->gu_scales_b + h->gu_bias_b + h->dn_codes_b +
                        h->dn_scales_b + h->dn_bias_b) / E);
}

int moe_last_launches(const moe_handle* h) { return h ? h->last_launches : 0; }

int moe_load_experts_ex(moe_handle* h, int layer, const void* gu_codes, const void* gu_scales,
                        const void* gu_bias, const void* dn_codes, const void* dn_scales,
                        const void* dn_bias, int flags, void* stream)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: handle is NULL");
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!gu_codes || !gu_scales || !dn_codes || !dn_scales)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: codes and scales must not be NULL");
    if (h->cfg.has_bias && (!gu_bias || !dn_bias))
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: has_bias=1 but a bias pointer is NULL");
    if (flags & ~(MOE_LOAD_GATE_UP_INTERLEAVED | MOE_LOAD_TRANSPOSED))
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts_ex: unknown flags 0x%x", flags);
    cudaStream_t s = (cudaStream_t)stream;
    const moe_config& c = h->cfg;
    const int H = c.hidden, I = c.intermediate, E = c.num_experts;
    const int blk = h->mxfp4 ? 32 : c.group, esz = h->mxfp4 ? 1 : 2;
    const bool ilv = (flags & MOE_LOAD_GATE_UP_INTERLEAVED) != 0, tr = (flags & MOE_LOAD_TRANSPOSED) != 0;
    uint8_t* base = h->arena + (size_t)layer * h->layer_stride;
    // the caller's tensors are copied to a staging area first (they may be host
    // memory), converted to the caller layout [N][K] with gate rows first if
    // the flags say they are in another one (a second area takes each
    // conversion's output), then reordered into the resident layout by a
    // repack kernel
    const size_t a_guc = align_up(h->gu_codes_b, 256), a_gus = align_up(h->gu_scales_b, 256);
    const size_t a_dnc = align_up(h->dn_codes_b, 256), a_dns = align_up(h->dn_scales_b, 256);
    const size_t a_gub = ilv && h->gu_bias_b ? align_up(h->gu_bias_b, 256) : 0;
    const size_t st_bytes = a_guc + a_gus + a_dnc + a_dns + a_gub;
    uint8_t* staging = nullptr;
    int rc = dev_alloc(&staging, flags ? 2 * st_bytes : st_bytes, "load staging");
    if (rc != MOE_OK)
        return rc;
    uint8_t* cur[4] = {staging, staging + a_guc, staging + a_guc + a_gus, staging + a_guc + a_gus + a_dnc};
    uint8_t* oth[4] = {cur[0] + st_bytes, cur[1] + st_bytes, cur[2] + st_bytes, cur[3] + st_bytes};
    uint8_t* st_gub = staging + a_guc + a_gus + a_dnc + a_dns;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(cur[0], gu_codes, h->gu_codes_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(cur[1], gu_scales, h->gu_scales_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(cur[2], dn_codes, h->dn_codes_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(cur[3], dn_scales, h->dn_scales_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (h->gu_bias_b && (e = cudaMemcpyAsync(a_gub ? st_gub : base + h->off_gu_bias, gu_bias, h->gu_bias_b,
                                              cudaMemcpyDefault, s)) != cudaSuccess) ||
        (h->dn_bias_b && (e = cudaMemcpyAsync(base + h->off_dn_bias, dn_bias, h->dn_bias_b,
                                              cudaMemcpyDefault, s)) != cudaSuccess)) {
        cudaStreamSynchronize(s);
        cudaFree(staging);
        return cuda_fail(e, "moe_load_experts copy");
    }
    auto flip = [&](int i) { uint8_t* t = cur[i]; cur[i] = oth[i]; oth[i] = t; };
    if (tr) {
        // [K][N] orientation: codes [E][K][N/2], scales [E][K/blk][N]
        if ((e = moe::launch_transpose_nibbles(cur[0], oth[0], E, 2 * I, H, s)) == cudaSuccess &&
            (e = moe::launch_transpose_elems(cur[1], oth[1], E, H / blk, 2 * I, esz, s)) == cudaSuccess &&
            (e = moe::launch_transpose_nibbles(cur[2], oth[2], E, H, I, s)) == cudaSuccess)
            e = moe::launch_transpose_elems(cur[3], oth[3], E, I / blk, H, esz, s);
        for (int i = 0; i < 4; ++i)
            flip(i);
    }
    if (e == cudaSuccess && ilv) {
        // gate row j at 2j, up row j at 2j + 1 (codes, scales and the gate/up bias)
        if ((e = moe::launch_deinterleave_rows(cur[0], oth[0], E, 2 * I, H / 2, s)) == cudaSuccess &&
            (e = moe::launch_deinterleave_rows(cur[1], oth[1], E, 2 * I, (long long)(H / blk) * esz, s)) ==
                cudaSuccess &&
            a_gub)
            e = moe::launch_deinterleave_rows(st_gub, base + h->off_gu_bias, E, 2 * I, 2, s);
        flip(0);
        flip(1);
    }
    if (e == cudaSuccess) {
        if (h->mxfp4) {
            // gate rows [0, I) and up rows [I, 2I) interleaved per 64 in 128-row tiles
            if ((e = moe::launch_repack_tiles(cur[0], cur[1], E, 2 * I, 2 * I, H, I, 0, base,
                                              (long long)h->gu_expert, s)) == cudaSuccess)
                e = moe::launch_repack_tiles(cur[2], cur[3], E, H, H, I, 0, 1, base + h->off_dn,
                                             (long long)h->dn_expert, s);
        } else {
            if ((e = moe::launch_repack_i4(cur[0], reinterpret_cast<const uint16_t*>(cur[1]), E, H, I, c.group, 0,
                                           base, (long long)h->gu_expert, s)) == cudaSuccess)
                e = moe::launch_repack_i4(cur[2], reinterpret_cast<const uint16_t*>(cur[3]), E, H, I, c.group, 1,
                                          base + h->off_dn, (long long)h->dn_expert, s);
        }
    }
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(s);
        cudaFree(staging);
        return cuda_fail(e, "moe_load_experts repack");
    }
    cudaFree(staging);
    h->loaded[layer] = 1;
    return MOE_OK;
}

int moe_load_experts(moe_handle* h, int layer, const void* gu_codes, const void* gu_scales,
                     const void* gu_bias, const void* dn_codes, const void* dn_scales,
                     const void* dn_bias, void* stream)
{
    return moe_load_experts_ex(h, layer, gu_codes, gu_scales, gu_bias, dn_codes, dn_scales, dn_bias, 0, stream);
}

int moe_forward(moe_handle* h, int layer, const void* x_bf16, const float* router_logits, int M,
                int top_k, void* out_bf16, void* stream)
{
    return forward_impl(h, layer, x_bf16, router_logits, M, top_k, out_bf16, nullptr, stream);
}

int moe_debug_forward_f32(moe_handle* h, int layer, const void* x_bf16, const float* router_logits, int M,
                          int top_k, void* out_bf16, float* out_f32, void* stream)
{
    if (!out_f32)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_forward_f32: out_f32 is NULL");
    if (reinterpret_cast<uintptr_t>(out_f32) & 15u)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_forward_f32: out_f32 must be 16-byte aligned");
    return forward_impl(h, layer, x_bf16, router_logits, M, top_k, out_bf16, out_f32, stream);
}

int moe_debug_set_wait(moe_handle* h, int spin_limit, int skip_cta)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_set_wait: handle is NULL");
    if (spin_limit < 0 || skip_cta < -1)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_set_wait: spin_limit must be >= 0, skip_cta >= -1");
    h->spin_limit = spin_limit == 0 ? moe::kSpinLimit : spin_limit;
    h->skip_cta = skip_cta;
    return MOE_OK;
}

int moe_forward_host(moe_handle* h, int layer, const void* x_bf16, const float* router_logits,
                     int M, int top_k, void* out_bf16, void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (!x_bf16 || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_host: x and out must not be NULL");
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!h->loaded[layer])
        return fail(MOE_ERR_NOT_LOADED, "moe_forward_host: layer %d has no experts loaded", layer);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = (size_t)M * h->cfg.hidden * 2, nl = (size_t)M * h->cfg.num_experts * 4;
    // x, the residual and the logits packed into the handle's mapped pinned
    // buffer by the host; the layer kernel reads them from there and writes the
    // result back there itself (no copy engine round trips: the pages' lesson
    // on per-token host work, keep it to a fixed, small amount).  The previous
    // call on this handle has completed (it synchronised before returning).
    std::memcpy(h->st_host, x_bf16, nb);
    std::memcpy(h->st_host + h->st_off_r, out_bf16, nb);
    if (router_logits)
        std::memcpy(h->st_host + h->st_off_l, router_logits, nl);
    rc = moe_forward(h, layer, h->st_dev,
                     router_logits ? reinterpret_cast<const float*>(h->st_dev + h->st_off_l) : nullptr, M, top_k,
                     h->st_dev + h->st_off_r, stream);
    if (rc != MOE_OK)
        return rc;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward_host");
    std::memcpy(out_bf16, h->st_host + h->st_off_r, nb);
    return MOE_OK;
}

int moe_forward_stack_steps(moe_handle* h, int n, void* resid_bf16, const float* router_logits, int M, int top_k,
                            void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (M > moe::kMaxTokens)
        return fail(MOE_ERR_UNSUPPORTED, "moe_forward_stack: M=%d > %d; the stack runs the decode kernel only", M,
                    moe::kMaxTokens);
    if (n < 1)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack_steps: n=%d must be >= 1", n);
    if (!resid_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack: resid must not be NULL");
    if (!aligned16(resid_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack: resid and logits must be 16-byte aligned");
    if ((rc = check_all_loaded(h, "moe_forward_stack")) != MOE_OK)
        return rc;
    const int L = h->cfg.num_layers;
    if (!router_logits && (rc = check_router(h, 0, L, "moe_forward_stack")) != MOE_OK)
        return rc;
    if ((long long)n * L > (1ll << 30))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack_steps: n * L = %lld layer calls is too many",
                    (long long)n * L);
    // the n x L layer calls in one persistent launch (grid barriers between them):
    // call c runs layer c mod L on step c / L's residual; each layer's input is the
    // normalised residual, which the kernel forms itself
    cudaError_t e = launch_seq(h, 0, n * L, router_logits, (long long)M * h->cfg.num_experts * sizeof(float),
                               nullptr, 0, resid_bf16, (long long)M * h->cfg.hidden * 2, nullptr, 0, M, top_k,
                               (cudaStream_t)stream, L);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward_stack launch");
    h->last_steps = n * L;
    h->last_first_layer = 0;
    h->last_launches = 1;
    return MOE_OK;
}

int moe_forward_stack(moe_handle* h, void* resid_bf16, const float* router_logits, int M, int top_k,
                      void* stream)
{
    return moe_forward_stack_steps(h, 1, resid_bf16, router_logits, M, top_k, stream);
}

int moe_forward_steps(moe_handle* h, int n, int layer0, const void* x_bf16, const float* router_logits, int M,
                      int top_k, void* out_bf16, void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (M > moe::kMaxTokens)
        return fail(MOE_ERR_UNSUPPORTED, "moe_forward_steps: M=%d > %d; decode sizes only", M, moe::kMaxTokens);
    const int L = h->cfg.num_layers;
    if (n < 1 || layer0 < 0 || layer0 >= L)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_steps: n=%d must be >= 1 and layer0=%d in 0..%d", n, layer0,
                    L - 1);
    if (!x_bf16 || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_steps: x and out must not be NULL");
    if (!aligned16(x_bf16) || !aligned16(out_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_steps: x, logits and out must be 16-byte aligned");
    if (!device_accessible(x_bf16) || (router_logits && !device_accessible(router_logits)) ||
        !device_accessible(out_bf16))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_steps: x, logits and out must be device memory or "
                                         "page-locked host memory mapped at the same address");
    const size_t nb = (size_t)n * M * h->cfg.hidden * 2;
    if (overlaps(x_bf16, nb, out_bf16, nb))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_steps: x overlaps out");
    for (int s = 0; s < n && s < L; ++s)
        if (!h->loaded[(layer0 + s) % L])
            return fail(MOE_ERR_NOT_LOADED, "moe_forward_steps: layer %d has no experts loaded", (layer0 + s) % L);
    if (!router_logits && (rc = check_router(h, layer0, n, "moe_forward_steps")) != MOE_OK)
        return rc;
    const long long xs = (long long)M * h->cfg.hidden * 2, ls = (long long)M * h->cfg.num_experts * sizeof(float);
    cudaError_t e = launch_seq(h, layer0, n, router_logits, ls, x_bf16, xs, out_bf16, xs, nullptr, 0, M, top_k,
                               (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward_steps launch");
    h->last_steps = n;
    h->last_first_layer = layer0;
    h->last_launches = 1;
    return MOE_OK;
}

int moe_debug_stack_trace(moe_handle* h, void* resid_bf16, const float* router_logits, int M,
                          int top_k, void* trace_bf16, void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (M > moe::kMaxTokens)
        return fail(MOE_ERR_UNSUPPORTED, "moe_debug_stack_trace: M=%d > %d; the stack runs the decode kernel only", M,
                    moe::kMaxTokens);
    if (!resid_bf16 || !trace_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stack_trace: NULL argument");
    if (!aligned16(resid_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stack_trace: resid and logits must be 16-byte aligned");
    if ((rc = check_all_loaded(h, "moe_debug_stack_trace")) != MOE_OK)
        return rc;
    if (!router_logits && (rc = check_router(h, 0, h->cfg.num_layers, "moe_debug_stack_trace")) != MOE_OK)
        return rc;
    const int L = h->cfg.num_layers;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = (size_t)M * h->cfg.hidden * 2;
    uint8_t* tr = static_cast<uint8_t*>(trace_bf16);
    cudaError_t e = cudaMemcpyAsync(tr, resid_bf16, nb, cudaMemcpyDeviceToDevice, s);
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        e = launch_decode(h, l, router_logits ? router_logits + (size_t)l * M * h->cfg.num_experts : nullptr,
                          nullptr, resid_bf16, M, top_k, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(tr + (size_t)(l + 1) * nb, resid_bf16, nb, cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_stack_trace");
    h->last_steps = L;
    h->last_first_layer = 0;
    h->last_launches = L;
    return MOE_OK;
}

int moe_load_router(moe_handle* h, int layer, const void* w_bf16, const void* bias_bf16)
{
    if (!h || !w_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_router: handle and weights must not be NULL");
    const moe_config& c = h->cfg;
    if (layer < 0 || layer >= c.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_router: layer=%d out of range 0..%d", layer, c.num_layers - 1);
    const size_t wb = (size_t)c.num_experts * c.hidden * 2, bb = (size_t)c.num_experts * 2;
    cudaError_t e;
    if (!h->rw) {
        h->rw_stride = align_up(wb + bb, 256);
        int rc = dev_alloc(&h->rw, h->rw_stride * c.num_layers, "router weights");
        if (rc != MOE_OK)
            return rc;
    }
    uint8_t* dst = h->rw + (size_t)layer * h->rw_stride;
    if ((e = cudaMemcpy(dst, w_bf16, wb, cudaMemcpyDefault)) != cudaSuccess ||
        (e = bias_bf16 ? cudaMemcpy(dst + wb, bias_bf16, bb, cudaMemcpyDefault) : cudaMemset(dst + wb, 0, bb)) !=
            cudaSuccess)
        return cuda_fail(e, "moe_load_router copy");
    h->rloaded[layer] = 1;
    return MOE_OK;
}

int moe_debug_router_logits(moe_handle* h, float* out_dev, int M, void* stream)
{
    if (!h || !out_dev)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_router_logits: NULL argument");
    if (M < 1 || M > std::max(h->cfg.max_tokens, moe::kMaxTokens))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_router_logits: M=%d out of range", M);
    cudaError_t e = cudaMemcpyAsync(out_dev, h->rlog, (size_t)M * h->cfg.num_experts * sizeof(float),
                                    cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_router_logits");
    return MOE_OK;
}

int moe_debug_stream_weights(moe_handle* h, int layer0, int n, long long bytes, void* stream)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stream_weights: handle is NULL");
    const int L = h->cfg.num_layers;
    if (layer0 < 0 || layer0 >= L || n < 1 || layer0 + n > L || bytes < 16 || bytes % 16 ||
        bytes > (long long)h->layer_stride)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stream_weights: need layers [layer0, layer0 + n) within 0..%d "
                    "and 16 <= bytes <= %zu, a multiple of 16", L - 1, h->layer_stride);
    cudaError_t e = moe::launch_stream_read(h->arena + (size_t)layer0 * h->layer_stride, (long long)h->layer_stride,
                                            bytes, n, h->cnt + 2, h->spin_limit, h->status, h->num_sms,
                                            (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_stream_weights launch");
    return MOE_OK;
}

int moe_set_batched_numerics(moe_handle* h, int numerics)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_set_batched_numerics: handle is NULL");
    if (numerics != MOE_BATCHED_MXFP4 && numerics != MOE_BATCHED_BF16)
        return fail(MOE_ERR_INVALID_ARG, "moe_set_batched_numerics: unknown numerics %d", numerics);
    if (!h->batched)
        return fail(MOE_ERR_UNSUPPORTED, "moe_set_batched_numerics: the handle has no batched path (max_tokens <= %d)",
                    moe::kMaxTokens);
    if (numerics == MOE_BATCHED_BF16 && !h->b_a16) {
        const moe_config& c = h->cfg;
        const size_t rows = (size_t)c.max_tokens * c.max_top_k + 16 * (size_t)h->max_tiles;
        int rc = dev_alloc(&h->b_a16, moe::batched_f16_act_bytes((long long)rows, c.hidden, c.intermediate),
                           "bf16 activation tiles");
        if (rc != MOE_OK)
            return rc;
        cudaError_t e = moe::prepare_batched_f16_kernels();
        if (e != cudaSuccess)
            return cuda_fail(e, "bf16 batched kernel set-up");
    }
    h->b_f16 = numerics == MOE_BATCHED_BF16 ? 1 : 0;
    return MOE_OK;
}

int moe_set_swiglu(moe_handle* h, float alpha, float limit, float beta)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_set_swiglu: handle is NULL");
    if (!std::isfinite(alpha) || !(limit > 0.0f) || std::isnan(limit) || !std::isfinite(beta))
        return fail(MOE_ERR_INVALID_ARG, "moe_set_swiglu: alpha and beta must be finite and limit > 0 (or +inf)");
    h->sw_alpha = alpha;
    h->sw_limit = limit;
    h->sw_beta = beta;
    return MOE_OK;
}

int moe_get_status(moe_handle* h, void* stream)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_get_status: handle is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    int st = 0;
    cudaError_t e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess ||
        (e = cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemset(h->status, 0, sizeof(int))) != cudaSuccess)
        return cuda_fail(e, "moe_get_status");
    if (st != MOE_OK) {
        // a call gave up waiting: its cross-CTA counters may be left part-way; clear
        // them (the call tags restart with the counters, so the flags are cleared too)
        if ((e = cudaMemset(h->cnt, 0, moe::kTcCounterWords * sizeof(unsigned long long))) != cudaSuccess ||
            (h->pflag && (e = cudaMemset(h->pflag, 0, (size_t)h->num_sms * sizeof(unsigned))) != cudaSuccess) ||
            (e = cudaDeviceSynchronize()) != cudaSuccess)
            return cuda_fail(e, "moe_get_status reset");
    }
    return st;
}

int moe_last_bytes(moe_handle* h, void* stream, long long* bytes)
{
    if (!h || !bytes)
        return fail(MOE_ERR_INVALID_ARG, "moe_last_bytes: NULL argument");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_last_bytes sync");
    const int L = h->cfg.num_layers;
    std::vector<int> nu(L, 0);
    if (h->last_steps > 0) {
        e = cudaMemcpy(nu.data(), h->stats, L * sizeof(int), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_last_bytes read");
    }
    long long total = 0;
    for (int s2 = 0; s2 < h->last_steps; ++s2)
        total += (long long)nu[(h->last_first_layer + s2) % L] * moe_expert_bytes(h);
    *bytes = total;
    return MOE_OK;
}

int moe_debug_dequant(moe_handle* h, int layer, int expert, int proj, float* out_dev, void* stream)
{
    if (!h || !out_dev)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_dequant: NULL argument");
    const moe_config& c = h->cfg;
    if (layer < 0 || layer >= c.num_layers || expert < 0 || expert >= c.num_experts ||
        (proj != 0 && proj != 1))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_dequant: layer/expert/proj out of range");
    if (!h->loaded[layer])
        return fail(MOE_ERR_NOT_LOADED, "moe_debug_dequant: layer %d has no experts loaded", layer);
    const int N = proj == 0 ? 2 * c.intermediate : c.hidden;
    const int K = proj == 0 ? c.hidden : c.intermediate;
    // the very bytes the forward kernels stream, decoded back to caller order
    const uint8_t* base = h->arena + (size_t)layer * h->layer_stride;
    const uint8_t* src = proj == 0 ? base + (size_t)expert * h->gu_expert
                                   : base + h->off_dn + (size_t)expert * h->dn_expert;
    cudaError_t e = h->mxfp4 ? moe::launch_dequant_tiles(src, N, K, proj == 0 ? c.intermediate : 0, proj, out_dev,
                                                         (cudaStream_t)stream)
                             : moe::launch_dequant_i4(src, c.hidden, c.intermediate, c.group, proj, out_dev,
                                                      (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_dequant launch");
    return MOE_OK;
}

int moe_debug_route(moe_handle* h, const float* logits, int M, int top_k, int* idx, float* w,
                    void* stream)
{
    if (!h || !logits || !idx || !w)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_route: NULL argument");
    if (M < 1 || M > 65536)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_route: M=%d must be in 1..65536", M);
    if (top_k < 1 || top_k > h->cfg.max_top_k)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_route: top_k=%d must be in 1..%d", top_k,
                    h->cfg.max_top_k);
    cudaError_t e = moe::launch_route(logits, M, h->cfg.num_experts, top_k, idx, w,
                                      (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_route launch");
    return MOE_OK;
}

int moe_debug_mx_quantize(const float* in, long long n, unsigned char* codes, unsigned char* scales,
                          void* stream)
{
    if (!in || !codes || !scales)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_mx_quantize: NULL argument");
    if (n < 0 || n % 32)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_mx_quantize: n=%lld must be a non-negative multiple of 32", n);
    if (!aligned16(in) || !aligned16(codes))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_mx_quantize: in and codes must be 16-byte aligned");
    cudaError_t e = moe::launch_mx_quantize(in, n, codes, scales, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_mx_quantize launch");
    return MOE_OK;
}

int moe_debug_batched_h(moe_handle* h, unsigned char* codes, unsigned char* scales, void* stream)
{
    if (!h || !codes || !scales)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_batched_h: NULL argument");
    if (!aligned16(codes))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_batched_h: codes must be 16-byte aligned");
    if (!h->batched || h->last_bM == 0)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_batched_h: no batched forward has run on this handle");
    moe::BatchParams b = batch_params(h, 0);
    b.M = h->last_bM;
    b.k = h->last_bk;
    cudaError_t e = moe::launch_untile_h(b, codes, scales, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_batched_h launch");
    return MOE_OK;
}

}  // extern "C"
