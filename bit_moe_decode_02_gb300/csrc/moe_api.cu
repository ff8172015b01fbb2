// moe_api.cu -- the C ABI declared in include/moe.h: handle, argument checks,
// resident weight arena, workspace, launch of the decode kernels and the
// cached CUDA graph of the expert stack.
//
// All tables the kernels need are fixed at moe_create / moe_load_experts; a
// forward call does no host-side work that depends on the routing (the pages'
// lesson: per-token host setup once cost 10.65 ms of a 36.95 ms token,
// "Amortizing the per-token host-sync setup tax ...", section 3), and it
// allocates nothing (the grow-only buffer cache that reallocated on every
// count change, TinyTitan tracker D114).
#include <cuda_runtime.h>

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

struct StackGraph {
    int M = 0, k = 0;
    const void* resid = nullptr;
    const void* logits = nullptr;
    cudaGraphExec_t exec = nullptr;
};

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
    // caller-layout tensor sizes in bytes (one layer, all experts)
    size_t gu_codes_b = 0, gu_scales_b = 0, gu_bias_b = 0;
    size_t dn_codes_b = 0, dn_scales_b = 0, dn_bias_b = 0;
    // resident layout: per layer [gate_up slabs][down slabs][gu bias][dn bias];
    // MXFP4 keeps no slabs (its kernels read the tile layout): [gu bias][dn bias]
    int sb = 0;                       // scale bytes per (segment, g) entry
    int gu_slab = 0, dn_slab = 0;     // bytes of one 16-row slab
    size_t gu_expert = 0, dn_expert = 0;
    size_t layer_stride = 0;
    size_t off_dn = 0, off_gu_bias = 0, off_dn_bias = 0;
    int slot_bytes = 0, nslots = 0, grid = 0;
    uint8_t* arena = nullptr;
    uint32_t* special = nullptr;      // [L][E][2]
    std::vector<char> loaded;
    // MXFP4: tile-layout copy of the weights (tensor-core decode and batched paths)
    bool tiles = false;
    bool batched = false;             // max_tokens > kMaxTokens
    size_t tc_smem = 0;
    float* tc_part = nullptr;
    float* tc_gpart = nullptr;      // split units: pieces' gate/up partial sums
    unsigned* tc_flags = nullptr;   // split units: [G] piece flags
    uint8_t* tc_xt = nullptr;
    unsigned long long* tc_cnt = nullptr;
    size_t t_gu_expert = 0, t_dn_expert = 0, t_off_dn = 0, t_layer_stride = 0;
    uint8_t* tarena = nullptr;
    int max_tiles = 0;
    int* b_int = nullptr;             // idx | slot | etile | erow | ntiles
    float* b_wt = nullptr;
    moe::TokTile* b_tiles = nullptr;
    uint8_t* b_xq = nullptr;
    uint8_t* b_xsf = nullptr;
    uint8_t* b_hq = nullptr;
    uint8_t* b_hsf = nullptr;
    float* b_y = nullptr;
    int last_bM = 0, last_bk = 0;     // M and top_k of the last batched call
    // workspace
    float* h = nullptr;
    float* ypart = nullptr;
    unsigned* counters = nullptr;     // done | hmax | slab_cnt | exit (see counter_words)
    int* stats = nullptr;   // distinct experts per layer of the last call
    int* status = nullptr;
    // staging for moe_forward_host: [x][residual / out][logits], on the device
    // and in pinned host memory, so one copy each way moves a call's data
    uint8_t* st_dev = nullptr;
    uint8_t* st_host = nullptr;
    size_t st_off_r = 0, st_off_l = 0, st_bytes = 0;
    // cross-CTA waits of the MXFP4 decode layer (moe_debug_set_wait)
    int spin_limit = moe::kSpinLimit;
    int skip_cta = -1;
    // stack graphs
    cudaStream_t capture_stream = nullptr;
    std::vector<StackGraph> graphs;
    int last_layers = 0;       // layers touched by the last forward call
    int last_first_layer = 0;
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
    for (auto& g : h->graphs)
        if (g.exec)
            cudaGraphExecDestroy(g.exec);
    if (h->capture_stream)
        cudaStreamDestroy(h->capture_stream);
    cudaFree(h->arena);
    cudaFree(h->special);
    cudaFree(h->h);
    cudaFree(h->ypart);
    cudaFree(h->counters);
    cudaFree(h->stats);
    cudaFree(h->status);
    cudaFree(h->st_dev);
    cudaFreeHost(h->st_host);
    cudaFree(h->tarena);
    cudaFree(h->tc_part);
    cudaFree(h->tc_gpart);
    cudaFree(h->tc_flags);
    cudaFree(h->tc_xt);
    cudaFree(h->tc_cnt);
    cudaFree(h->b_int);
    cudaFree(h->b_wt);
    cudaFree(h->b_tiles);
    cudaFree(h->b_xq);
    cudaFree(h->b_xsf);
    cudaFree(h->b_hq);
    cudaFree(h->b_hsf);
    cudaFree(h->b_y);
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

// Token capacity of the decode kernel's workspace and shared memory.
int decode_tokens(const moe_config& c)
{
    return c.max_tokens < moe::kMaxTokens ? c.max_tokens : moe::kMaxTokens;
}

moe::LayerParams layer_params(const moe_handle* h, int layer)
{
    const moe_config& c = h->cfg;
    const uint8_t* base = h->arena + (size_t)layer * h->layer_stride;
    moe::LayerParams p{};
    p.gu = base;
    p.dn = base + h->off_dn;
    p.gu_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(base + h->off_gu_bias) : nullptr;
    p.dn_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(base + h->off_dn_bias) : nullptr;
    p.special = h->special + (size_t)layer * c.num_experts * 2;
    p.h = h->h;
    p.ypart = h->ypart;
    p.done = h->counters;
    p.hmax = h->counters + moe::kMaxUnits;
    p.slab_cnt = p.hmax + moe::kMaxUnits * moe::kMaxTokens;
    p.exit_cnt = p.slab_cnt + c.hidden / moe::kSlabRows;
    p.status = h->status;
    p.nu_out = h->stats + layer;
    p.gu_expert_bytes = (long long)h->gu_expert;
    p.dn_expert_bytes = (long long)h->dn_expert;
    p.gu_slab_bytes = h->gu_slab;
    p.dn_slab_bytes = h->dn_slab;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.kmax = c.max_top_k;
    p.mmax = decode_tokens(c);
    p.group = c.group;
    p.nslots = h->nslots;
    p.slot_bytes = h->slot_bytes;
    return p;
}

// MXFP4: tile-layout weights and the workspace of the tensor-core decode kernel.
int create_tiles(moe_handle* h)
{
    const moe_config& c = h->cfg;
    const int H = c.hidden, I = c.intermediate, E = c.num_experts;
    h->tiles = true;
    h->t_gu_expert = (size_t)moe::tile_proj_bytes(2 * I, H);   // interleaved gate_up
    h->t_dn_expert = (size_t)moe::tile_proj_bytes(H, I);
    h->t_off_dn = align_up(E * h->t_gu_expert, 256);
    h->t_layer_stride = align_up(h->t_off_dn + E * h->t_dn_expert, 256);
    const int G = h->num_sms;
    int rc;
    if ((rc = dev_alloc(&h->tarena, h->t_layer_stride * c.num_layers, "tile-layout weights")) ||
        (rc = dev_alloc(&h->tc_part, moe::tc_part_bytes(G, H), "per-CTA outputs")) ||
        (rc = dev_alloc(&h->tc_gpart, (size_t)G * moe::kRowTile * 4 * sizeof(float), "split-unit partials")) ||
        (rc = dev_alloc(&h->tc_flags, (size_t)G * sizeof(unsigned), "split-unit flags")) ||
        (rc = dev_alloc(&h->tc_xt, moe::tc_terms_bytes(H), "x terms")) ||
        (rc = dev_alloc(&h->tc_cnt, moe::kTcCounterWords * sizeof(unsigned long long), "counters")))
        return rc;
    cudaError_t e = cudaMemset(h->tc_cnt, 0, moe::kTcCounterWords * sizeof(unsigned long long));
    // x-term rows past M * 8 are never written and feed MMA columns nobody reads:
    // keep them zero (valid E2M1 codes, E8M0 byte 0) instead of leftover bytes
    if (e == cudaSuccess)
        e = cudaMemset(h->tc_xt, 0, moe::tc_terms_bytes(H));
    if (e == cudaSuccess)
        e = cudaMemset(h->tc_flags, 0, (size_t)G * sizeof(unsigned));
    if (e != cudaSuccess)
        return cuda_fail(e, "counters");
    // all the shared memory a block may have: the kernel's own plus the stage ring
    int dev = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return cuda_fail(e, "shared memory limit");
    h->tc_smem = (size_t)optin - moe::decode_tc_static_smem();
    if ((e = moe::prepare_decode_tc(h->tc_smem)) != cudaSuccess)
        return cuda_fail(e, "tensor-core decode kernel set-up");
    return MOE_OK;
}

moe::DecodeTcParams tc_params(const moe_handle* h, int layer)
{
    const moe_config& c = h->cfg;
    const uint8_t* tb = h->tarena + (size_t)layer * h->t_layer_stride;
    const uint8_t* sb = h->arena + (size_t)layer * h->layer_stride;
    moe::DecodeTcParams p{};
    p.gu = tb;
    p.dn = tb + h->t_off_dn;
    p.gu_expert = (long long)h->t_gu_expert;
    p.dn_expert = (long long)h->t_dn_expert;
    p.gu_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(sb + h->off_gu_bias) : nullptr;
    p.dn_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(sb + h->off_dn_bias) : nullptr;
    p.part = h->tc_part;
    p.gpart = h->tc_gpart;
    p.pflag = h->tc_flags;
    p.xt = h->tc_xt;
    p.xcnt = h->tc_cnt;
    p.done = h->tc_cnt + 1;
    p.status = h->status;
    p.nu_out = h->stats + layer;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.smem_bytes = (int)h->tc_smem;
    p.spin_limit = h->spin_limit;
    p.skip_cta = h->skip_cta;
    return p;
}

// Kernel launches of one decode layer: the layer kernel (tensor-core MXFP4 or int4).
int decode_launches(const moe_handle*) { return 1; }

// The decode layer on the current kernel of this handle's format; out_f32
// (debug, nullable) also receives the result before its bf16 rounding.
cudaError_t launch_decode(const moe_handle* h, int layer, const float* logits, const void* x, void* resid,
                          int M, int k, cudaStream_t s, float* out_f32 = nullptr)
{
    if (h->tiles) {
        moe::DecodeTcParams p = tc_params(h, layer);
        p.logits = logits;
        p.x = static_cast<const uint16_t*>(x);
        p.resid = static_cast<uint16_t*>(resid);
        p.out_f32 = out_f32;
        p.M = M;
        p.k = k;
        return moe::launch_decode_tc(p, h->tc_smem, h->num_sms, s);
    }
    moe::LayerParams p = layer_params(h, layer);
    p.logits = logits;
    p.x = static_cast<const uint16_t*>(x);
    p.resid = static_cast<uint16_t*>(resid);
    p.out_f32 = out_f32;
    p.M = M;
    p.k = k;
    return moe::launch_layer(p, h->cfg.format, h->grid, s);
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
    const uint8_t* tb = h->tarena + (size_t)layer * h->t_layer_stride;
    const uint8_t* sb = h->arena + (size_t)layer * h->layer_stride;
    moe::BatchParams p{};
    p.gu = tb;
    p.dn = tb + h->t_off_dn;
    p.gu_expert = (long long)h->t_gu_expert;
    p.dn_expert = (long long)h->t_dn_expert;
    p.gu_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(sb + h->off_gu_bias) : nullptr;
    p.dn_bias = c.has_bias ? reinterpret_cast<const uint16_t*>(sb + h->off_dn_bias) : nullptr;
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
    p.status = h->status;
    p.nu_out = h->stats + layer;
    p.H = c.hidden;
    p.I = c.intermediate;
    p.E = c.num_experts;
    p.max_tiles = h->max_tiles;
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

// Caller layout -> tile layout for one layer (gate rows [0, I) and up rows
// [I, 2I) of gate_up become two projections of I rows each).
cudaError_t load_tiles(moe_handle* h, int layer, const uint8_t* guc, const uint8_t* gus,
                       const uint8_t* dnc, const uint8_t* dns, cudaStream_t s)
{
    const moe_config& c = h->cfg;
    const int H = c.hidden, I = c.intermediate, E = c.num_experts;
    uint8_t* tb = h->tarena + (size_t)layer * h->t_layer_stride;
    cudaError_t e;
    if ((e = moe::launch_repack_tiles(guc, gus, E, 2 * I, 2 * I, H, I, tb, (long long)h->t_gu_expert, s)) !=
        cudaSuccess)
        return e;
    return moe::launch_repack_tiles(dnc, dns, E, H, H, I, 0, tb + h->t_off_dn, (long long)h->t_dn_expert, s);
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
    const size_t sbh = c.format == MOE_FMT_MXFP4 ? H / 32 : 2 * H / c.group;
    const size_t sbi = c.format == MOE_FMT_MXFP4 ? I / 32 : 2 * I / c.group;
    h->gu_codes_b = E * 2 * I * H / 2;
    h->gu_scales_b = E * 2 * I * sbh;
    h->gu_bias_b = c.has_bias ? E * 2 * I * 2 : 0;
    h->dn_codes_b = E * H * I / 2;
    h->dn_scales_b = E * H * sbi;
    h->dn_bias_b = c.has_bias ? E * H * 2 : 0;
    const bool slabs = c.format == MOE_FMT_INT4;   // MXFP4 weights live in the tile layout only
    h->sb = moe::scale_entry_bytes(c.format, c.group);
    if (slabs) {
        h->gu_slab = moe::slab_bytes((int)H, h->sb);
        h->dn_slab = moe::slab_bytes((int)I, h->sb);
        h->gu_expert = (2 * I / moe::kSlabRows) * (size_t)h->gu_slab;
        h->dn_expert = (H / moe::kSlabRows) * (size_t)h->dn_slab;
    }
    size_t off = align_up(E * h->gu_expert, 256);
    h->off_dn = off;
    off = align_up(off + E * h->dn_expert, 256);
    h->off_gu_bias = off;
    off = align_up(off + h->gu_bias_b, 256);
    h->off_dn_bias = off;
    off = align_up(off + h->dn_bias_b, 256);
    h->layer_stride = off > 256 ? off : 256;
    if (slabs) {
        h->slot_bytes = (int)align_up((size_t)(h->gu_slab > h->dn_slab ? h->gu_slab : h->dn_slab), 128);
        h->nslots = (int)((moe::kSmemBudget - moe::kRedBytes - moe::kXfragBytes -
                           2 * (size_t)decode_tokens(c) * I * sizeof(float)) / h->slot_bytes);
        if (h->nslots > moe::kMaxSlots)
            h->nslots = moe::kMaxSlots;
        if (h->nslots < 2) {
            free_handle(h);
            return fail(MOE_ERR_UNSUPPORTED, "a 16-row weight slab (%d bytes) is too large for the "
                        "shared-memory ring", h->slot_bytes);
        }
    }

    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "cudaGetDevice");
    }
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    h->grid = h->num_sms;   // one CTA per SM: every CTA of a layer is resident at once
    if (slabs) {
        int per_sm = 0;
        moe::LayerParams lp{};
        lp.nslots = h->nslots;
        lp.slot_bytes = h->slot_bytes;
        lp.mmax = decode_tokens(c);
        lp.I = c.intermediate;
        e = moe::prepare_layer_kernel(c.format, c.group, moe::layer_smem_bytes(lp), &per_sm);
        if (e != cudaSuccess) {
            free_handle(h);
            return cuda_fail(e, "layer kernel set-up");
        }
        if (per_sm < 1) {
            free_handle(h);
            return fail(MOE_ERR_UNSUPPORTED, "the layer kernel does not fit on an SM");
        }
    }
    const size_t Mx = c.max_tokens, Kx = c.max_top_k, Md = decode_tokens(c);
    const size_t ncount = moe::counter_words((int)H);
    h->st_off_r = align_up(Mx * H * 2, 256);
    h->st_off_l = h->st_off_r + align_up(Mx * H * 2, 256);
    h->st_bytes = h->st_off_l + Mx * E * sizeof(float);
    if ((rc = dev_alloc(&h->arena, h->layer_stride * c.num_layers, "expert weights")) ||
        (rc = dev_alloc(&h->special, (size_t)c.num_layers * E * 2 * sizeof(uint32_t), "flags")) ||
        (rc = dev_alloc(&h->h, Md * Kx * I * sizeof(float), "h workspace")) ||
        (rc = dev_alloc(&h->ypart, Md * Kx * H * sizeof(float), "y workspace")) ||
        (rc = dev_alloc(&h->counters, ncount * sizeof(unsigned), "counters")) ||
        (rc = dev_alloc(&h->stats, c.num_layers * sizeof(int), "stats")) ||
        (rc = dev_alloc(&h->status, sizeof(int), "status")) ||
        (rc = dev_alloc(&h->st_dev, h->st_bytes, "staging"))) {
        free_handle(h);
        return rc;
    }
    if ((e = cudaHostAlloc((void**)&h->st_host, h->st_bytes, cudaHostAllocDefault)) != cudaSuccess) {
        cudaGetLastError();
        h->st_host = nullptr;
        free_handle(h);
        return fail(MOE_ERR_OOM, "cudaHostAlloc(%zu bytes) for the host staging failed", h->st_bytes);
    }
    if ((e = cudaMemset(h->counters, 0, ncount * sizeof(unsigned))) != cudaSuccess ||
        (e = cudaMemset(h->special, 0, (size_t)c.num_layers * E * 2 * sizeof(uint32_t))) != cudaSuccess ||
        (e = cudaMemset(h->stats, 0, c.num_layers * sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(h->status, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "moe_create setup");
    }
    if ((c.format == MOE_FMT_MXFP4 && (rc = create_tiles(h)) != MOE_OK) ||
        (c.max_tokens > moe::kMaxTokens && (rc = create_batched(h)) != MOE_OK)) {
        free_handle(h);
        return rc;
    }
    h->loaded.assign(c.num_layers, 0);
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

int moe_load_experts(moe_handle* h, int layer, const void* gu_codes, const void* gu_scales,
                     const void* gu_bias, const void* dn_codes, const void* dn_scales,
                     const void* dn_bias, void* stream)
{
    if (!h)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: handle is NULL");
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!gu_codes || !gu_scales || !dn_codes || !dn_scales)
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: codes and scales must not be NULL");
    if (h->cfg.has_bias && (!gu_bias || !dn_bias))
        return fail(MOE_ERR_INVALID_ARG, "moe_load_experts: has_bias=1 but a bias pointer is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    const moe_config& c = h->cfg;
    uint8_t* base = h->arena + (size_t)layer * h->layer_stride;
    uint8_t* staging = nullptr;
    const size_t st_bytes = align_up(h->gu_codes_b, 256) + align_up(h->gu_scales_b, 256) +
                            align_up(h->dn_codes_b, 256) + align_up(h->dn_scales_b, 256);
    int rc = dev_alloc(&staging, st_bytes, "load staging");
    if (rc != MOE_OK)
        return rc;
    uint8_t* st_guc = staging;
    uint8_t* st_gus = st_guc + align_up(h->gu_codes_b, 256);
    uint8_t* st_dnc = st_gus + align_up(h->gu_scales_b, 256);
    uint8_t* st_dns = st_dnc + align_up(h->dn_codes_b, 256);
    uint32_t* special = h->special + (size_t)layer * c.num_experts * 2;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(st_guc, gu_codes, h->gu_codes_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(st_gus, gu_scales, h->gu_scales_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(st_dnc, dn_codes, h->dn_codes_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(st_dns, dn_scales, h->dn_scales_b, cudaMemcpyDefault, s)) != cudaSuccess ||
        (h->gu_bias_b && (e = cudaMemcpyAsync(base + h->off_gu_bias, gu_bias, h->gu_bias_b,
                                              cudaMemcpyDefault, s)) != cudaSuccess) ||
        (h->dn_bias_b && (e = cudaMemcpyAsync(base + h->off_dn_bias, dn_bias, h->dn_bias_b,
                                              cudaMemcpyDefault, s)) != cudaSuccess) ||
        (e = cudaMemsetAsync(special, 0, (size_t)c.num_experts * 2 * sizeof(uint32_t), s)) != cudaSuccess ||
        (!h->tiles && (e = moe::launch_repack(c.format, c.group, st_guc, st_gus, c.num_experts, 2 * c.intermediate,
                                              c.hidden, base, (long long)h->gu_expert, h->gu_slab, special, 0,
                                              s)) != cudaSuccess) ||
        (!h->tiles && (e = moe::launch_repack(c.format, c.group, st_dnc, st_dns, c.num_experts, c.hidden,
                                              c.intermediate, base + h->off_dn, (long long)h->dn_expert,
                                              h->dn_slab, special, 1, s)) != cudaSuccess) ||
        (h->tiles && (e = load_tiles(h, layer, st_guc, st_gus, st_dnc, st_dns, s)) != cudaSuccess) ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess) {
        cudaStreamSynchronize(s);
        cudaFree(staging);
        return cuda_fail(e, "moe_load_experts");
    }
    cudaFree(staging);
    h->loaded[layer] = 1;
    return MOE_OK;
}

}  // extern "C"

namespace {

int forward_impl(moe_handle* h, int layer, const void* x_bf16, const float* router_logits, int M,
                 int top_k, void* out_bf16, float* out_f32, void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!x_bf16 || !router_logits || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x, logits and out must not be NULL");
    if (!aligned16(x_bf16) || !aligned16(out_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x, logits and out must be 16-byte aligned");
    const size_t nb = (size_t)M * h->cfg.hidden * 2;
    if (overlaps(x_bf16, nb, out_bf16, nb))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: x overlaps out");
    if (!h->loaded[layer])
        return fail(MOE_ERR_NOT_LOADED, "moe_forward: layer %d has no experts loaded", layer);
    if (M > moe::kMaxTokens) {
        moe::BatchParams b = batch_params(h, layer);
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
        h->last_layers = 1;
        h->last_first_layer = layer;
        h->last_launches = launches;
        h->last_bM = M;
        h->last_bk = top_k;
        return MOE_OK;
    }
    cudaError_t e = launch_decode(h, layer, router_logits, x_bf16, out_bf16, M, top_k, (cudaStream_t)stream,
                                  out_f32);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward launch");
    h->last_layers = 1;
    h->last_first_layer = layer;
    h->last_launches = decode_launches(h);
    return MOE_OK;
}

}  // namespace

extern "C" {

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
    if (!x_bf16 || !router_logits || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_host: x, logits and out must not be NULL");
    if (layer < 0 || layer >= h->cfg.num_layers)
        return fail(MOE_ERR_INVALID_ARG, "layer=%d out of range 0..%d", layer, h->cfg.num_layers - 1);
    if (!h->loaded[layer])
        return fail(MOE_ERR_NOT_LOADED, "moe_forward_host: layer %d has no experts loaded", layer);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = (size_t)M * h->cfg.hidden * 2, nl = (size_t)M * h->cfg.num_experts * 4;
    // x, the residual and the logits packed into the handle's pinned staging
    // buffer by the host, so that one copy moves them; one copy brings the
    // result back (the pages' lesson on per-token host work: keep it to a
    // fixed, small amount)
    std::memcpy(h->st_host, x_bf16, nb);
    std::memcpy(h->st_host + h->st_off_r, out_bf16, nb);
    std::memcpy(h->st_host + h->st_off_l, router_logits, nl);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(h->st_dev, h->st_host, h->st_off_l + nl, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "moe_forward_host upload");
    rc = moe_forward(h, layer, h->st_dev, reinterpret_cast<const float*>(h->st_dev + h->st_off_l), M, top_k,
                     h->st_dev + h->st_off_r, stream);
    if (rc != MOE_OK)
        return rc;
    if ((e = cudaMemcpyAsync(h->st_host + h->st_off_r, h->st_dev + h->st_off_r, nb, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return cuda_fail(e, "moe_forward_host download");
    std::memcpy(out_bf16, h->st_host + h->st_off_r, nb);
    return MOE_OK;
}

int moe_forward_stack(moe_handle* h, void* resid_bf16, const float* router_logits, int M, int top_k,
                      void* stream)
{
    int rc = check_forward_args(h, M, top_k);
    if (rc != MOE_OK)
        return rc;
    if (M > moe::kMaxTokens)
        return fail(MOE_ERR_UNSUPPORTED, "moe_forward_stack: M=%d > %d; the stack runs the decode kernel only", M,
                    moe::kMaxTokens);
    if (!resid_bf16 || !router_logits)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack: resid and logits must not be NULL");
    if (!aligned16(resid_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_stack: resid and logits must be 16-byte aligned");
    const int L = h->cfg.num_layers;
    for (int l = 0; l < L; ++l)
        if (!h->loaded[l])
            return fail(MOE_ERR_NOT_LOADED, "moe_forward_stack: layer %d has no experts loaded", l);
    StackGraph* g = nullptr;
    for (auto& c : h->graphs)
        if (c.M == M && c.k == top_k && c.resid == resid_bf16 && c.logits == router_logits)
            g = &c;
    if (!g) {
        // capture the 2L launches once for this (M, top_k, buffers)
        cudaStream_t cs = h->capture_stream;
        cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_forward_stack capture begin");
        cudaError_t le = cudaSuccess;
        for (int l = 0; l < L && le == cudaSuccess; ++l)
            le = launch_decode(h, l, router_logits + (size_t)l * M * h->cfg.num_experts, nullptr, resid_bf16, M,
                               top_k, cs);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(cs, &graph);
        if (le != cudaSuccess || e != cudaSuccess) {
            if (graph)
                cudaGraphDestroy(graph);
            return cuda_fail(le != cudaSuccess ? le : e, "moe_forward_stack capture");
        }
        cudaGraphExec_t exec = nullptr;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_forward_stack instantiate");
        if (h->graphs.size() >= 8) {
            cudaGraphExecDestroy(h->graphs.front().exec);
            h->graphs.erase(h->graphs.begin());
        }
        StackGraph ng;
        ng.M = M;
        ng.k = top_k;
        ng.resid = resid_bf16;
        ng.logits = router_logits;
        ng.exec = exec;
        h->graphs.push_back(ng);
        g = &h->graphs.back();
    }
    cudaError_t e = cudaGraphLaunch(g->exec, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_forward_stack launch");
    h->last_layers = L;
    h->last_first_layer = 0;
    h->last_launches = L * decode_launches(h);
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
    if (!resid_bf16 || !router_logits || !trace_bf16)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stack_trace: NULL argument");
    if (!aligned16(resid_bf16) || !aligned16(router_logits))
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_stack_trace: resid and logits must be 16-byte aligned");
    const int L = h->cfg.num_layers;
    for (int l = 0; l < L; ++l)
        if (!h->loaded[l])
            return fail(MOE_ERR_NOT_LOADED, "moe_debug_stack_trace: layer %d has no experts loaded", l);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = (size_t)M * h->cfg.hidden * 2;
    uint8_t* tr = static_cast<uint8_t*>(trace_bf16);
    cudaError_t e = cudaMemcpyAsync(tr, resid_bf16, nb, cudaMemcpyDeviceToDevice, s);
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        e = launch_decode(h, l, router_logits + (size_t)l * M * h->cfg.num_experts, nullptr, resid_bf16, M, top_k,
                          s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(tr + (size_t)(l + 1) * nb, resid_bf16, nb, cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "moe_debug_stack_trace");
    h->last_layers = L;
    h->last_first_layer = 0;
    h->last_launches = L * decode_launches(h);
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
        // a call gave up waiting: its cross-CTA counters may be left part-way; clear them
        const size_t ncount = moe::counter_words(h->cfg.hidden);
        // (the call tags restart with the counters, so the flags are cleared too)
        if ((h->tc_cnt && (e = cudaMemset(h->tc_cnt, 0, moe::kTcCounterWords * sizeof(unsigned long long))) != cudaSuccess) ||
            (h->tc_flags && (e = cudaMemset(h->tc_flags, 0, (size_t)h->num_sms * sizeof(unsigned))) != cudaSuccess) ||
            (e = cudaMemset(h->counters, 0, ncount * sizeof(unsigned))) != cudaSuccess ||
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
    std::vector<int> nu(h->last_layers > 0 ? h->last_layers : 1, 0);
    if (h->last_layers > 0) {
        e = cudaMemcpy(nu.data(), h->stats + h->last_first_layer, h->last_layers * sizeof(int),
                       cudaMemcpyDeviceToHost);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_last_bytes read");
    }
    long long total = 0;
    for (int l = 0; l < h->last_layers; ++l)
        total += (long long)nu[l] * moe_expert_bytes(h);
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
    if (h->tiles) {
        // the bytes the tensor-core kernels stream (interleaved gate/up tiles,
        // scale chunks in tensor-memory order), decoded back to caller order
        const uint8_t* tb = h->tarena + (size_t)layer * h->t_layer_stride;
        const uint8_t* src = proj == 0 ? tb + (size_t)expert * h->t_gu_expert
                                       : tb + h->t_off_dn + (size_t)expert * h->t_dn_expert;
        cudaError_t e = moe::launch_dequant_tiles(src, N, K, proj == 0 ? c.intermediate : 0, out_dev,
                                                  (cudaStream_t)stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "moe_debug_dequant launch");
        return MOE_OK;
    }
    moe::LayerParams p = layer_params(h, layer);
    const uint8_t* slabs = proj == 0 ? p.gu + (size_t)expert * h->gu_expert
                                     : p.dn + (size_t)expert * h->dn_expert;
    cudaError_t e = moe::launch_dequant(c.format, c.group, slabs, N, K, proj == 0 ? h->gu_slab : h->dn_slab,
                                        out_dev, (cudaStream_t)stream);
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
