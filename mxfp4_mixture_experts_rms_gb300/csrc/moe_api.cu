// moe_api.cu -- the C-ABI of include/moe.h: plan, argument checks, workspace
// carving, weight registration and the per-forward launch sequence.
//
// Error conventions follow goosedump gpt_oss.rs, where every shape mismatch or
// out-of-range route is an `Err` (`ensure!` in `mixture_of_experts_batch`,
// `mix_expert_outputs`, the tensor validation): here every violation is a
// negative status with a message, never a crash.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "moe_common.cuh"

bool decode_supported(const BlockParams &bp);
cudaError_t launch_absmax(const float *v, int n, uint32_t *out, cudaStream_t st);

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// The thread's last-error message, for the other translation units.
int moe_fail_status(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}
void moe_set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

namespace {

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

constexpr int kMaxTokens = 65535;  // tokens per forward: one combine grid row each

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

}  // namespace

struct moe_plan {
    BlockParams bp;
    int max_tokens = 4096;
    int decode_max_tokens = -1;  // -1: chosen from the shape (auto_decode_max)
    int path = 0;
    int router_exact = 0;
    int stall_test = 0;              // test hook: the gate/up GEMV waits on a barrier nothing completes
    int noalloc_dev = -1;            // device of this plan's last moe_forward_noalloc (-1: none)
    void *ws_ptr = nullptr;
    size_t ws_bytes = 0;
    Workspace ws{};
    bool have_ws = false;
    bool have_w = false;
    moe_weights w{};
    MatPtrs gate{}, up{}, down{};
    PrefillMaps maps{};
    bool have_maps = false;
    uint8_t *pf_scales = nullptr;    // owned: the scales repacked for the grouped GEMM
    size_t pf_scales_bytes = 0;
    // the decode GEMVs carry x_hat / h as fp16 unless these can leave its range
    bool x_bf16 = false, h_bf16 = false;
    // the grouped GEMM takes fp16 operands (exponents in [104, 140], fp16-range activations)
    bool pf_f16 = false;
    // FP4 activations: the grouped GEMM on the block-scaled FP4 tensor cores (kind::mxf4)
    bool act_fp4 = false;
    bool out_bf16 = false;  // out receives bf16 (the next stacked block's input) instead of fp32
    moe_locality *loc = nullptr;  // attached locality profiler: every forward's routes are recorded
    int loc_layer = 0;
    long long loc_pos = 0;        // position of the next forward's first token
    Mxf4Weights mxf4{};
    bool have_mxf4 = false;
    uint8_t *mxf4_scales = nullptr;  // owned: weight scales repacked into the kernel's atoms
    size_t mxf4_scales_bytes = 0;
    // expert cache (expert_cache_slots > 0): the expert matrices stay in the
    // caller's store and `cache_slots` of them at a time in device slots
    int cache_slots = 0;
    MatPtrs src_gate{}, src_up{}, src_down{};  // the store's matrices (device-accessible views)
    void *cache_mem = nullptr;       // owned: the slots' arrays, the shared expert's copy, the tables
    CacheTables cache{};
    CacheArrays carr{};
    // kernel timing (profile option)
    static constexpr int kSlots = 4, kMaxRec = 4096 * kSlots;
    std::vector<cudaEvent_t> ev;     // 2 events per record
    std::vector<int> rec_slot;       // slot of each pending record
    bool profile = false;
};

namespace {

struct Carve {
    size_t off = 0;
    template <class T>
    T *take(char *base, size_t n) {
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off = align256(off + n * sizeof(T));
        return p;
    }
};

// Lays out and clears the expert cache: C slots of each of the nine arrays
// (codes, scales and biases of gate, up and down), a device copy of the shared
// expert, and the tables; the GEMVs then read the slots (and the shared
// expert's copy), the copy kernel the store.
int cache_setup(moe_plan *p) {
    const BlockParams &b = p->bp;
    const int C = p->cache_slots, E = b.E;
    const MatPtrs *src[3] = {&p->src_gate, &p->src_up, &p->src_down};
    size_t sz[kCacheArrays];
    for (int m = 0; m < 3; m++) {
        const size_t rows = (size_t)src[m]->rows, cols = (size_t)src[m]->cols;
        sz[3 * m] = rows * cols / 2;         // codes (a multiple of 16 bytes: cols % 32 == 0)
        sz[3 * m + 1] = rows * (cols / 32);  // scales (rows % 16 == 0)
        sz[3 * m + 2] = rows * 4;            // biases
    }
    long long W = 0;  // 16-byte words per expert
    for (int a = 0; a < kCacheArrays; a++) W += (long long)(sz[a] / 16);
    if ((long long)E * W >= (1LL << 31) - (1LL << 24))
        return fail(MOE_ESHAPE, "expert cache: %d experts of %lld bytes exceed the copy kernel's 32-bit word range",
                    E, W * 16);
    uint8_t *slot[kCacheArrays], *shc[kCacheArrays];
    Carve c;
    auto layout = [&](char *base) {
        c.off = 0;
        for (int a = 0; a < kCacheArrays; a++) slot[a] = c.take<uint8_t>(base, (size_t)C * sz[a]);
        for (int a = 0; a < kCacheArrays; a++) shc[a] = b.n_shared ? c.take<uint8_t>(base, sz[a]) : nullptr;
        p->cache.slot_of = c.take<int32_t>(base, E);
        p->cache.expert_of = c.take<int32_t>(base, C);
        p->cache.stamp = c.take<long long>(base, C);
        p->cache.miss = c.take<int2>(base, E);
        p->cache.n_miss = c.take<int32_t>(base, 1);
        p->cache.stats = c.take<long long>(base, 3);
        p->cache.fwd = c.take<long long>(base, 1);
    };
    layout(nullptr);
    if (p->cache_mem) {
        cudaFree(p->cache_mem);
        p->cache_mem = nullptr;
    }
    cudaError_t e = cudaMalloc(&p->cache_mem, c.off);
    if (e != cudaSuccess) {
        p->cache_mem = nullptr;
        return cuda_fail(e, "moe_load_weights (expert cache slots)");
    }
    layout(static_cast<char *>(p->cache_mem));
    p->cache.slots = C;
    // no expert resident, every slot empty (stamp -1), counters at zero
    e = cudaMemset(p->cache.slot_of, 0xFF, sizeof(int32_t) * E);
    if (e == cudaSuccess) e = cudaMemset(p->cache.expert_of, 0xFF, sizeof(int32_t) * C);
    if (e == cudaSuccess) e = cudaMemset(p->cache.stamp, 0xFF, sizeof(long long) * C);
    if (e == cudaSuccess) e = cudaMemset(p->cache.n_miss, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(p->cache.stats, 0, sizeof(long long) * 3);
    if (e == cudaSuccess) e = cudaMemset(p->cache.fwd, 0, sizeof(long long));
    const void *store[kCacheArrays], *shared[kCacheArrays];
    for (int m = 0; m < 3; m++) {
        store[3 * m] = src[m]->codes;
        store[3 * m + 1] = src[m]->scales;
        store[3 * m + 2] = src[m]->bias;
        shared[3 * m] = src[m]->sh_codes;
        shared[3 * m + 1] = src[m]->sh_scales;
        shared[3 * m + 2] = src[m]->sh_bias;
    }
    for (int a = 0; a < kCacheArrays && b.n_shared && e == cudaSuccess; a++)
        e = cudaMemcpy(shc[a], shared[a], sz[a], cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(e, "moe_load_weights (expert cache setup)");
    for (int a = 0; a < kCacheArrays; a++) {
        p->carr.src[a] = static_cast<const uint4 *>(store[a]);
        p->carr.dst[a] = reinterpret_cast<uint4 *>(slot[a]);
        p->carr.words[a] = (long long)(sz[a] / 16);
    }
    MatPtrs *dst[3] = {&p->gate, &p->up, &p->down};
    for (int m = 0; m < 3; m++) {
        dst[m]->codes = slot[3 * m];
        dst[m]->scales = slot[3 * m + 1];
        dst[m]->bias = reinterpret_cast<const float *>(slot[3 * m + 2]);
        dst[m]->sh_codes = shc[3 * m];
        dst[m]->sh_scales = shc[3 * m + 1];
        dst[m]->sh_bias = reinterpret_cast<const float *>(shc[3 * m + 2]);
    }
    return MOE_OK;
}

// Largest token count for which the GEMVs beat the grouped GEMM, measured on a
// GB300: with 32 experts the GEMV path wins up to 56 tokens and ties at 64
// (each expert tile then streams its weights with few routes per tile either
// way); with 256 experts it wins up to 8 tokens, the grouped GEMM from 12.
int auto_decode_max(const BlockParams &b) { return b.E <= 64 ? 60 : 8; }

// Which projection kernels run for this token count: the GEMV (decode) path
// or the tensor-core grouped GEMM (prefill) path.
int choose_path(const moe_plan *p, int tokens, bool *decode, int *nt, int *tile_rows) {
    const BlockParams &b = p->bp;
    if (p->act_fp4) {
        // FP4 activations: the block-scaled FP4 grouped GEMM at every token count
        if (!p->have_mxf4) return fail(MOE_ESHAPE, "the FP4-activation path needs H and F multiples of 64, H <= 4096");
        *decode = false;
        *nt = 1;
        *tile_rows = prefill_tile_rows();
        return MOE_OK;
    }
    // the grouped GEMM needs H and F in whole 64-element stages; the GEMVs need
    // H, F <= 4480 (register-resident activations)
    const bool prefill_ok = b.H % 64 == 0 && b.F % 64 == 0 && p->have_maps;
    const bool decode_ok = decode_supported(b);
    if (p->path == 2 && !prefill_ok) return fail(MOE_ESHAPE, "the prefill path needs H and F multiples of 64");
    if (p->path == 1 && !decode_ok) return fail(MOE_ESHAPE, "the decode path needs H and F <= 4480");
    const int dmax = p->decode_max_tokens >= 0 ? p->decode_max_tokens : auto_decode_max(b);
    bool d = p->path == 1 || (p->path == 0 && (!prefill_ok || (decode_ok && tokens <= dmax)));
    if (d && !decode_ok) return fail(MOE_ESHAPE, "no kernel path for H=%d F=%d", b.H, b.F);
    *decode = d;
    // 8-route GEMV tiles up to 32 tokens (measured on a GB300: the 16-token
    // 24-layer stack runs 2.12 ms per step with them against 3.09 ms with
    // 16-route tiles, whose larger split-K partials leave one stage fewer in
    // flight); an expert with more routes takes several tiles
    *nt = tokens <= 32 ? 1 : 2;
    *tile_rows = d ? 8 * *nt : prefill_tile_rows();
    return MOE_OK;
}

int max_tiles_for(const moe_plan *p, int T) {
    // T <= kMaxTokens and K + n_shared <= 9 keep this far inside int
    const size_t R = (size_t)T * (p->bp.K + p->bp.n_shared);
    return (int)(R / 8 + 2 * (size_t)(p->bp.E + p->bp.n_shared) + 8);
}

// Lays the workspace out for T tokens; with base == nullptr only sizes it.
size_t carve(const moe_plan *p, int T, char *base, Workspace *ws) {
    const BlockParams &b = p->bp;
    const size_t R = (size_t)T * (b.K + b.n_shared);
    Carve c;
    Workspace w{};
    w.xhat = c.take<uint16_t>(base, (size_t)T * b.H);
    w.xhat_mma = c.take<uint16_t>(base, (size_t)T * b.H);
    w.xhat16 = c.take<uint16_t>(base, (size_t)T * b.H);
    w.ids = c.take<int32_t>(base, (size_t)T * b.K);
    w.route_w = c.take<float>(base, (size_t)T * b.K);
    w.counts = c.take<int32_t>(base, b.E + 1);
    w.offsets = c.take<int32_t>(base, b.E + 2);
    w.perm_token = c.take<int32_t>(base, R);
    w.perm_slot = c.take<int32_t>(base, R);
    w.perm_w = c.take<float>(base, R);
    w.loc = c.take<int32_t>(base, R);
    w.max_tiles = max_tiles_for(p, T);
    w.tiles = c.take<int4>(base, w.max_tiles);
    w.n_tiles = c.take<int32_t>(base, 4);
    w.h = c.take<uint16_t>(base, R * b.F);
    w.h16 = c.take<uint16_t>(base, R * b.F);
    w.y = c.take<float>(base, R * b.H);
    w.xs = reinterpret_cast<uint16_t *>(w.y);
    w.logits = c.take<float>(base, (size_t)T * b.E);
    w.lbound = c.take<float>(base, (size_t)T * b.E);
    w.xnorm = c.take<float>(base, (size_t)T);
    w.wnorm = c.take<float>(base, (size_t)b.E);
    w.status = c.take<int32_t>(base, 4);
    w.tickets = c.take<uint32_t>(base, route_ticket_count(T));
    if (p->act_fp4) {
        // FP4 operands: codes alias buffers the FP4 path does not otherwise use
        // (x_hat codes are dead before y is written; h16 is the bf16 paths');
        // scale atoms per 128-route tile
        w.xq = reinterpret_cast<uint8_t *>(w.y);
        w.hq = reinterpret_cast<uint8_t *>(w.h16);
        const size_t tiles = R / 128 + (size_t)(b.E + b.n_shared) + 2;
        w.xsf = c.take<uint8_t>(base, tiles * mxf4_nqe(b.H) * 512);
        w.hsf = c.take<uint8_t>(base, tiles * mxf4_nqe(b.F) * 512);
    }
    if (ws) *ws = w;
    return c.off;
}

MatPtrs mat_of(const moe_mxfp4_matrix &m, const moe_mxfp4_matrix &sh, int rows, int cols) {
    MatPtrs r;
    r.codes = m.codes;
    r.scales = m.scales;
    r.bias = m.bias;
    r.sh_codes = sh.codes;
    r.sh_scales = sh.scales;
    r.sh_bias = sh.bias;
    r.rows = rows;
    r.cols = cols;
    return r;
}

// The optional per-token outputs of a forward: the routing kernel writes ids
// and route weights with 4-byte stores and x_hat with 16-byte stores, while it
// still reads x.
int check_outputs(const BlockParams &b, int tokens, const uint16_t *x, const int32_t *ids_out, const float *rw_out,
                  const uint16_t *xhat_out) {
    if (!aligned4(ids_out) || !aligned4(rw_out))
        return fail(MOE_EINVAL, "ids and route-weight outputs must be 4-byte aligned");
    if (!aligned16(xhat_out)) return fail(MOE_EINVAL, "the x_hat output must be 16-byte aligned");
    const char *xb = reinterpret_cast<const char *>(x), *hb = reinterpret_cast<const char *>(xhat_out);
    const size_t n = (size_t)tokens * b.H * 2;
    if (hb && hb < xb + n && xb < hb + n) return fail(MOE_EINVAL, "the x_hat output must not overlap x");
    return MOE_OK;
}

// A view of p the kernels can read: device memory, or pinned / registered host
// memory (its device mapping); null where the device cannot reach p.
const void *device_view(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.devicePointer;
}

// The store's matrix m as the kernels see it (MOE_EINVAL where a pointer is not device-accessible).
int store_view(const moe_mxfp4_matrix &m, const char *name, moe_mxfp4_matrix *out) {
    out->codes = static_cast<const uint8_t *>(device_view(m.codes));
    out->scales = static_cast<const uint8_t *>(device_view(m.scales));
    out->bias = static_cast<const float *>(device_view(m.bias));
    if (!out->codes || !out->scales || !out->bias)
        return fail(MOE_EINVAL, "%s: with expert_cache_slots the expert matrices must be device memory or pinned "
                    "(page-locked) host memory", name);
    if (!aligned16(out->codes) || !aligned16(out->scales) || !aligned16(out->bias))
        return fail(MOE_EINVAL, "%s: pointers must be 16-byte aligned", name);
    return MOE_OK;
}

int check_matrix(const moe_mxfp4_matrix &m, const char *name) {
    if (!m.codes || !m.scales || !m.bias) return fail(MOE_EINVAL, "%s: NULL pointer", name);
    if (!aligned16(m.codes) || !aligned16(m.scales) || !aligned16(m.bias))
        return fail(MOE_EINVAL, "%s: pointers must be 16-byte aligned", name);
    return MOE_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Forward without any allocation: the workspace lives in a static device array.
// Some callers cannot allocate device memory -- a runtime that owns every byte
// of device memory through its own pool and forbids cudaMalloc, or code that
// must not risk the implicit device synchronisation an allocation can cause.
// For them the same kernels run on a fixed scratch array that every GPU
// loading this library reserves once, at module load, until exit.  Its first
// 256 bytes are the status word of the kernels run on it (read and cleared by
// moe_get_device_status); the workspace is carved from the rest.
#define MOE_NOALLOC_SCRATCH_BYTES (16u << 20)
#define MOE_NOALLOC_STATUS_BYTES 256u
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[256];  // device address of g_noalloc_scratch, per device ordinal

// The device address of the static scratch array on device `dev`, looked up
// once per device with that device current (in host code the array's name is
// only a host-side stand-in, not a device address).
int noalloc_scratch_addr(int dev, void **out) {
    if (dev < 0 || dev >= 256) return fail(MOE_EINVAL, "moe_forward_noalloc: device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "moe_forward_noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}
// The launch sequence of one forward on workspace ws: routing (+ permutation),
// gate/up, down, combine.  mark(slot, begin) brackets each kernel slot (the
// profile option's events; a no-op otherwise).
template <class Mark>
int enqueue_forward(moe_plan *p, const Workspace &ws, const uint16_t *x, int tokens, float *out, int32_t *ids_out,
                    float *rw_out, uint16_t *xhat_out, cudaStream_t st, Mark &&mark) {
    const BlockParams &b = p->bp;
    bool decode = false;
    int nt = 1, tile_rows = 0;
    if (int rc = choose_path(p, tokens, &decode, &nt, &tile_rows)) return rc;
    const bool cached = p->cache_slots > 0;
    if (cached) {
        // every expert a forward routes to must have a slot at once
        if (!decode) return fail(MOE_ESHAPE, "the expert cache serves the decode GEMVs; %d tokens take another path", tokens);
        const long long reach = std::min<long long>(b.E, (long long)tokens * b.K);
        if (reach > p->cache_slots)
            return fail(MOE_ESHAPE, "%d tokens can route to %lld experts; the expert cache holds %d", tokens, reach,
                        p->cache_slots);
    }
    mark(0, true);
    const int forms = p->act_fp4 ? 0 : decode ? (p->x_bf16 ? 0 : kFormF16) : (p->pf_f16 ? kFormF16 : kFormMma);
    cudaError_t e = launch_route(b, ws, x, p->w.gamma, p->w.router_w, p->w.router_b, tokens, ids_out, rw_out,
                                 xhat_out, tile_rows, p->router_exact, forms, st);
    // the expert cache: slots for the routed experts, the missing ones copied in
    if (cached && e == cudaSuccess) e = launch_cache_assign(p->cache, b, ws, st);
    if (cached && e == cudaSuccess) e = launch_cache_copy(p->cache, p->carr, st);
    mark(0, false);
    if (e != cudaSuccess) return cuda_fail(e, "routing kernel launch");
    mark(1, true);
    if (p->act_fp4) {
        e = launch_mxf4_stage(b, ws, p->gate, p->up, p->down, p->mxf4, tokens, true, st);
    } else {
        if (!decode) e = launch_gather(b, ws, tokens, p->pf_f16, st);
        if (e == cudaSuccess)
            e = decode ? launch_decode_stage(b, ws, p->gate, p->up, true, tokens, nt, p->x_bf16, p->h_bf16,
                                             p->stall_test, cached, st)
                       : launch_prefill_stage(b, ws, p->gate, p->up, true, tokens, p->maps.gateup, p->pf_f16, st);
    }
    mark(1, false);
    if (e != cudaSuccess) return cuda_fail(e, "gate/up kernel launch");
    mark(2, true);
    if (p->act_fp4)
        e = launch_mxf4_stage(b, ws, p->gate, p->up, p->down, p->mxf4, tokens, false, st);
    else
        e = decode ? launch_decode_stage(b, ws, p->down, p->down, false, tokens, nt, p->x_bf16, p->h_bf16, 0, cached,
                                         st)
                   : launch_prefill_stage(b, ws, p->down, p->down, false, tokens, p->maps.down, p->pf_f16, st);
    mark(2, false);
    if (e != cudaSuccess) return cuda_fail(e, "down kernel launch");
    mark(3, true);
    e = launch_combine(b, ws, x, tokens, out, p->out_bf16 ? 1 : 0, st);
    mark(3, false);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    if (p->loc) {
        e = locality_enqueue(p->loc, p->loc_layer, ws.ids, ws.route_w, tokens, p->loc_pos, st);
        if (e != cudaSuccess) return cuda_fail(e, "locality profiler launch");
        p->loc_pos += tokens;
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_last_error(void) { return g_err; }

int moe_locality_attach(moe_plan *p, moe_locality *prof, int layer) {
    if (!p) return fail(MOE_EINVAL, "NULL plan");
    if (prof && layer < 0) return fail(MOE_EINVAL, "layer must be >= 0");
    p->loc = prof;
    p->loc_layer = layer;
    p->loc_pos = 0;
    return MOE_OK;
}

moe_plan *moe_plan_create(int hidden, int expert_hidden, int n_experts, int top_k, float swiglu_alpha,
                          float swiglu_limit, float weight_scale) {
    if (hidden <= 0 || hidden % 32 || expert_hidden <= 0 || expert_hidden % 32) {
        fail(MOE_ESHAPE, "hidden and expert_hidden must be positive multiples of 32 (got %d, %d)", hidden,
             expert_hidden);
        return nullptr;
    }
    if (n_experts < 1 || n_experts > MOE_MAX_EXPERTS) {
        fail(MOE_ESHAPE, "n_experts must be in [1, %d] (got %d)", MOE_MAX_EXPERTS, n_experts);
        return nullptr;
    }
    if (top_k < 1 || top_k > n_experts || top_k > MOE_MAX_TOPK) {
        fail(MOE_ESHAPE, "top_k must be in [1, min(n_experts, %d)] (got %d)", MOE_MAX_TOPK, top_k);
        return nullptr;
    }
    if (!(swiglu_limit > 0.f) || !(swiglu_alpha == swiglu_alpha) || !(weight_scale == weight_scale)) {
        fail(MOE_EINVAL, "swiglu_limit must be > 0 and alpha, weight_scale finite");
        return nullptr;
    }
    moe_plan *p = new (std::nothrow) moe_plan();
    if (!p) {
        fail(MOE_ENOMEM, "out of host memory");
        return nullptr;
    }
    p->bp.H = hidden;
    p->bp.F = expert_hidden;
    p->bp.E = n_experts;
    p->bp.K = top_k;
    p->bp.n_shared = 0;
    p->bp.alpha = swiglu_alpha;
    p->bp.limit = swiglu_limit;
    p->bp.wscale = weight_scale;
    p->bp.eps = 1e-5;
    g_err[0] = 0;
    return p;
}

void moe_plan_destroy(moe_plan *plan) {
    if (!plan) return;
    for (auto &e : plan->ev) cudaEventDestroy(e);
    if (plan->pf_scales) cudaFree(plan->pf_scales);
    if (plan->mxf4_scales) cudaFree(plan->mxf4_scales);
    if (plan->cache_mem) cudaFree(plan->cache_mem);
    delete plan;
}

int moe_plan_set_i(moe_plan *p, const char *key, long long v) {
    if (!p || !key) return fail(MOE_EINVAL, "NULL plan or key");
    if (!strcmp(key, "n_shared_experts")) {
        if (v != 0 && v != 1) return fail(MOE_EINVAL, "n_shared_experts must be 0 or 1");
        if (p->have_ws) return fail(MOE_EINVAL, "n_shared_experts must be set before moe_set_workspace");
        p->bp.n_shared = (int)v;
        p->have_w = false;
    } else if (!strcmp(key, "max_tokens")) {
        // the combine kernel takes one grid row per token (grid y <= 65535)
        if (v < 1 || v > kMaxTokens) return fail(MOE_EINVAL, "max_tokens must be in [1, %d]", kMaxTokens);
        if (p->have_ws) return fail(MOE_EINVAL, "max_tokens must be set before moe_set_workspace");
        p->max_tokens = (int)v;
    } else if (!strcmp(key, "decode_max_tokens")) {
        if (v < -1 || v > (1 << 20)) return fail(MOE_EINVAL, "decode_max_tokens out of range");
        p->decode_max_tokens = (int)v;
    } else if (!strcmp(key, "path")) {
        if (v < 0 || v > 2) return fail(MOE_EINVAL, "path must be 0, 1 or 2");
        p->path = (int)v;
    } else if (!strcmp(key, "router_exact")) {
        p->router_exact = v ? 1 : 0;
    } else if (!strcmp(key, "out_bf16")) {
        p->out_bf16 = v != 0;
    } else if (!strcmp(key, "act_fp4")) {
        if (p->have_ws) return fail(MOE_EINVAL, "act_fp4 must be set before moe_set_workspace");
        p->act_fp4 = v != 0;
        p->have_w = false;  // the weights are prepared for the path at load
    } else if (!strcmp(key, "expert_cache_slots")) {
        if (v < 0 || v > p->bp.E) return fail(MOE_EINVAL, "expert_cache_slots must be in [0, n_experts]");
        p->cache_slots = (int)v;
        p->have_w = false;  // the slots are laid out at load
    } else if (!strcmp(key, "test_stall_wait")) {
        p->stall_test = v ? 1 : 0;
    } else if (!strcmp(key, "profile")) {
        if (v && p->ev.empty()) {
            p->ev.resize(2 * moe_plan::kMaxRec);
            for (auto &e : p->ev)
                if (cudaEventCreate(&e) != cudaSuccess) return fail(MOE_ECUDA, "cudaEventCreate failed");
        }
        p->profile = v != 0;
        p->rec_slot.clear();
    } else {
        return fail(MOE_EINVAL, "unknown integer option '%s'", key);
    }
    return MOE_OK;
}

int moe_plan_path_for(const moe_plan *p, int tokens) {
    if (!p) return fail(MOE_EINVAL, "NULL plan");
    if (!p->have_w) return fail(MOE_ENOTREADY, "moe_load_weights has not been called");
    bool decode = false;
    int nt = 1, tile_rows = 0;
    const int rc = choose_path(p, tokens, &decode, &nt, &tile_rows);
    if (rc != MOE_OK) return rc;
    return p->act_fp4 ? 3 : decode ? 1 : 2;
}

int moe_plan_set_f(moe_plan *p, const char *key, double v) {
    if (!p || !key) return fail(MOE_EINVAL, "NULL plan or key");
    if (!strcmp(key, "rms_eps")) {
        if (!(v >= 0.0)) return fail(MOE_EINVAL, "rms_eps must be >= 0");
        p->bp.eps = v;
    } else {
        return fail(MOE_EINVAL, "unknown floating option '%s'", key);
    }
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_plan *p, int max_tokens) {
    if (!p) {
        fail(MOE_EINVAL, "NULL plan");
        return 0;
    }
    int T = max_tokens > 0 ? max_tokens : p->max_tokens;
    if (T > kMaxTokens) {
        fail(MOE_EINVAL, "max_tokens %d > %d", T, kMaxTokens);
        return 0;
    }
    return carve(p, T, nullptr, nullptr);
}

int moe_set_workspace(moe_plan *p, void *dev_ptr, size_t bytes) {
    if (!p || !dev_ptr) return fail(MOE_EINVAL, "NULL plan or workspace");
    if (((uintptr_t)dev_ptr & 255u) != 0) return fail(MOE_EINVAL, "workspace must be 256-byte aligned");
    size_t need = carve(p, p->max_tokens, nullptr, nullptr);
    if (bytes < need) return fail(MOE_ENOMEM, "workspace too small: %zu < %zu bytes", bytes, need);
    carve(p, p->max_tokens, static_cast<char *>(dev_ptr), &p->ws);
    cudaError_t e = cudaMemset(p->ws.status, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(p->ws.tickets, 0, sizeof(uint32_t) * route_ticket_count(p->max_tokens));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "moe_set_workspace");
    p->ws_ptr = dev_ptr;
    p->ws_bytes = bytes;
    p->have_ws = true;
    return MOE_OK;
}

int moe_load_weights(moe_plan *p, const moe_weights *w) {
    if (!p || !w) return fail(MOE_EINVAL, "NULL plan or weights");
    if (!w->gamma || !w->router_w || !w->router_b) return fail(MOE_EINVAL, "NULL gamma/router pointer");
    if (!aligned16(w->gamma) || !aligned16(w->router_w) || !aligned16(w->router_b))
        return fail(MOE_EINVAL, "gamma/router pointers must be 16-byte aligned");
    int rc;
    if ((rc = check_matrix(w->gate, "gate")) || (rc = check_matrix(w->up, "up")) ||
        (rc = check_matrix(w->down, "down")))
        return rc;
    if (p->bp.n_shared) {
        if ((rc = check_matrix(w->sh_gate, "sh_gate")) || (rc = check_matrix(w->sh_up, "sh_up")) ||
            (rc = check_matrix(w->sh_down, "sh_down")))
            return rc;
    }
    if (p->cache_slots && p->act_fp4)
        return fail(MOE_EINVAL, "the expert cache serves the decode GEMVs: act_fp4 cannot be combined with it");
    // with the expert cache the expert matrices may live in host memory: the
    // kernels read them through their device views
    moe_weights wd = *w;
    if (p->cache_slots) {
        if ((rc = store_view(w->gate, "gate", &wd.gate)) || (rc = store_view(w->up, "up", &wd.up)) ||
            (rc = store_view(w->down, "down", &wd.down)))
            return rc;
        if (p->bp.n_shared &&
            ((rc = store_view(w->sh_gate, "sh_gate", &wd.sh_gate)) || (rc = store_view(w->sh_up, "sh_up", &wd.sh_up)) ||
             (rc = store_view(w->sh_down, "sh_down", &wd.sh_down))))
            return rc;
        w = &wd;
    }
    const BlockParams &b = p->bp;
    // reject the NaN scale code (0xFF) up front
    int32_t *flag = nullptr;
    cudaError_t e = cudaMalloc(&flag, 8);
    if (e != cudaSuccess) return cuda_fail(e, "moe_load_weights");
    e = cudaMemset(flag, 0, 4);
    const size_t n_gu = (size_t)b.F * (b.H / 32), n_d = (size_t)b.H * (b.F / 32);
    const moe_mxfp4_matrix *ms[6] = {&w->gate, &w->up, &w->down, &w->sh_gate, &w->sh_up, &w->sh_down};
    for (int i = 0; i < (b.n_shared ? 6 : 3) && e == cudaSuccess; i++) {
        size_t n = (i % 3 == 2 ? n_d : n_gu) * (i < 3 ? b.E : 1);
        e = launch_scan_scales(ms[i]->scales, n, flag, 0);
    }
    // max |gamma| (second word of the flag buffer) bounds |x_hat| <= sqrt(H) max|gamma|
    if (e == cudaSuccess) e = cudaMemset(flag + 1, 0, 4);
    if (e == cudaSuccess) e = launch_absmax(w->gamma, b.H, reinterpret_cast<uint32_t *>(flag + 1), 0);
    int32_t h[2] = {0, 0};
    if (e == cudaSuccess) e = cudaMemcpy(h, flag, 8, cudaMemcpyDeviceToHost);
    cudaFree(flag);
    if (e != cudaSuccess) return cuda_fail(e, "moe_load_weights scale scan");
    if (h[0] & 1) return fail(MOE_EINVAL, "an E8M0 scale holds the NaN code 0xFF");
    float gmax;
    memcpy(&gmax, &h[1], 4);
    p->w = *w;
    p->gate = mat_of(w->gate, w->sh_gate, b.F, b.H);
    p->up = mat_of(w->up, w->sh_up, b.F, b.H);
    p->down = mat_of(w->down, w->sh_down, b.H, b.F);
    p->src_gate = p->gate;
    p->src_up = p->up;
    p->src_down = p->down;
    p->have_maps = false;
    p->have_mxf4 = false;
    if (p->cache_slots) {
        // the GEMVs read the slots (no grouped-GEMM preparation: the cache
        // serves the decode path)
        if ((rc = cache_setup(p))) return rc;
    } else if (b.H % 64 == 0 && b.F % 64 == 0 &&
               prefill_make_maps(b, p->gate, p->up, p->down, &p->maps) == cudaSuccess) {
        const size_t nbytes = prefill_scales_bytes(b);
        if (p->pf_scales && p->pf_scales_bytes != nbytes) {
            cudaFree(p->pf_scales);
            p->pf_scales = nullptr;
        }
        if (!p->pf_scales) {
            e = cudaMalloc(&p->pf_scales, nbytes);
            if (e != cudaSuccess) {
                p->pf_scales = nullptr;
                return cuda_fail(e, "moe_load_weights (repacked scales)");
            }
            p->pf_scales_bytes = nbytes;
        }
        e = prefill_pack_scales(b, p->gate, p->up, p->down, p->pf_scales, &p->maps, 0);
        if (e == cudaSuccess) e = cudaStreamSynchronize(0);
        if (e != cudaSuccess) return cuda_fail(e, "moe_load_weights (repacked scales)");
        p->have_maps = true;
    }
    if (p->act_fp4 && b.H % 64 == 0 && b.F % 64 == 0 && b.H <= 4096) {
        const size_t nbytes = mxf4_scales_bytes(b);
        if (p->mxf4_scales && p->mxf4_scales_bytes != nbytes) {
            cudaFree(p->mxf4_scales);
            p->mxf4_scales = nullptr;
        }
        if (!p->mxf4_scales) {
            e = cudaMalloc(&p->mxf4_scales, nbytes);
            if (e != cudaSuccess) {
                p->mxf4_scales = nullptr;
                return cuda_fail(e, "moe_load_weights (FP4 scale atoms)");
            }
            p->mxf4_scales_bytes = nbytes;
        }
        e = mxf4_prepare(b, p->gate, p->up, p->down, p->mxf4_scales, &p->mxf4, 0);
        if (e == cudaSuccess) e = cudaStreamSynchronize(0);
        if (e != cudaSuccess) return cuda_fail(e, "moe_load_weights (FP4 scale atoms)");
        p->have_mxf4 = true;
    }
    // fp16 holds the GEMV activations below 65504: |x_hat| <= sqrt(H) max|gamma|;
    // |h| <= max(|L|, 0.3/alpha) (|L| + 1), since x sigmoid(alpha x) >= -0.28/alpha
    const double xb = std::sqrt((double)b.H) * (double)gmax * 1.01;
    const double L = std::fabs((double)b.limit);
    const double gb = b.alpha > 0.f ? std::max(L, 0.3 / (double)b.alpha) : INFINITY;
    const double hb = gb * (L + 1.0) * 1.01;
    p->x_bf16 = !(xb < 65504.0);
    p->h_bf16 = !(hb < 65504.0);
    p->pf_f16 = !(h[0] & 2) && !p->x_bf16 && !p->h_bf16;
    p->have_w = true;
    return MOE_OK;
}

int moe_forward_ex(moe_plan *p, const uint16_t *x, int tokens, float *out, int32_t *ids_out, float *rw_out,
                   uint16_t *xhat_out, void *stream) {
    if (!p) return fail(MOE_EINVAL, "NULL plan");
    if (tokens < 0) return fail(MOE_EINVAL, "tokens must be >= 0");
    if (tokens == 0) return MOE_OK;
    if (!x || !out) return fail(MOE_EINVAL, "NULL x or out");
    if (!p->have_w) return fail(MOE_ENOTREADY, "moe_load_weights has not been called");
    if (!p->have_ws) return fail(MOE_ENOTREADY, "moe_set_workspace has not been called");
    if (tokens > p->max_tokens) return fail(MOE_ENOMEM, "tokens %d > max_tokens %d", tokens, p->max_tokens);
    if (!aligned16(x) || !aligned16(out)) return fail(MOE_EINVAL, "x and out must be 16-byte aligned");
    const BlockParams &b = p->bp;
    const char *xb = reinterpret_cast<const char *>(x), *ob = reinterpret_cast<const char *>(out);
    if (xb < ob + (size_t)tokens * b.H * (p->out_bf16 ? 2 : 4) && ob < xb + (size_t)tokens * b.H * 2)
        return fail(MOE_EINVAL, "x and out must not alias");
    if (int rc = check_outputs(b, tokens, x, ids_out, rw_out, xhat_out)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto mark = [&](int slot, bool begin) {
        if (!p->profile) return;
        if (begin) {
            if ((int)p->rec_slot.size() >= moe_plan::kMaxRec) return;
            p->rec_slot.push_back(slot);
            // external record: becomes an event node when the forward is graph-captured
            cudaEventRecordWithFlags(p->ev[2 * (p->rec_slot.size() - 1)], st, cudaEventRecordExternal);
        } else if (!p->rec_slot.empty() && p->rec_slot.back() == slot) {
            cudaEventRecordWithFlags(p->ev[2 * (p->rec_slot.size() - 1) + 1], st, cudaEventRecordExternal);
        }
    };
    return enqueue_forward(p, p->ws, x, tokens, out, ids_out, rw_out, xhat_out, st, mark);
}

int moe_forward(moe_plan *p, const uint16_t *x, int tokens, float *out, int32_t *ids_out, void *stream) {
    return moe_forward_ex(p, x, tokens, out, ids_out, nullptr, nullptr, stream);
}

int moe_get_expert_counts(const moe_plan *p, int32_t *dev_counts_out, void *stream) {
    if (!p || !dev_counts_out) return fail(MOE_EINVAL, "NULL argument");
    if (!p->have_ws) return fail(MOE_ENOTREADY, "no workspace");
    cudaError_t e = cudaMemcpyAsync(dev_counts_out, p->ws.counts, sizeof(int32_t) * p->bp.E,
                                    cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_get_expert_counts");
}

int moe_get_permutation(const moe_plan *p, int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                        void *stream) {
    if (!p || !offsets || !perm_token || !perm_slot) return fail(MOE_EINVAL, "NULL argument");
    if (!p->have_ws) return fail(MOE_ENOTREADY, "no workspace");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int EE = p->bp.E + p->bp.n_shared;
    // route count of the last forward = offsets[EE]; copy the maximum extent
    const size_t R = (size_t)p->max_tokens * (p->bp.K + p->bp.n_shared);
    cudaError_t e = cudaMemcpyAsync(offsets, p->ws.offsets, sizeof(int32_t) * (EE + 1), cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(perm_token, p->ws.perm_token, sizeof(int32_t) * R, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(perm_slot, p->ws.perm_slot, sizeof(int32_t) * R, cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_get_permutation");
}

int moe_debug_dequant(const moe_plan *p, int expert, int which, float *dev_out, void *stream) {
    if (!p || !dev_out) return fail(MOE_EINVAL, "NULL argument");
    if (!p->have_w) return fail(MOE_ENOTREADY, "moe_load_weights has not been called");
    if (which < 0 || which > 2) return fail(MOE_EINVAL, "which must be 0 (gate), 1 (up) or 2 (down)");
    if (!aligned4(dev_out)) return fail(MOE_EINVAL, "dev_out must be 4-byte aligned");
    if (expert < 0 || expert > p->bp.E || (expert == p->bp.E && !p->bp.n_shared))
        return fail(MOE_EINVAL, "expert %d out of range", expert);
    const MatPtrs &m = which == 0 ? p->src_gate : which == 1 ? p->src_up : p->src_down;  // the store
    cudaError_t e = launch_dequant(m, expert, p->bp.E, dev_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_debug_dequant");
}

int moe_get_cache_state(const moe_plan *p, int32_t *slot_of, long long *stats, void *stream) {
    if (!p) return fail(MOE_EINVAL, "NULL plan");
    if (!p->cache_slots || !p->have_w || !p->cache_mem)
        return fail(MOE_ENOTREADY, "the plan has no expert cache (expert_cache_slots, then moe_load_weights)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (slot_of) e = cudaMemcpyAsync(slot_of, p->cache.slot_of, sizeof(int32_t) * p->bp.E, cudaMemcpyDeviceToHost, st);
    if (stats && e == cudaSuccess)
        e = cudaMemcpyAsync(stats, p->cache.stats, sizeof(long long) * 3, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_get_cache_state");
}

int moe_profile_read(moe_plan *p, double *total_ms, int *launches, int n_slots) {
    if (!p || !total_ms || !launches || n_slots < 0) return fail(MOE_EINVAL, "NULL argument");
    for (int i = 0; i < n_slots; i++) {
        total_ms[i] = 0.0;
        launches[i] = 0;
    }
    for (size_t r = 0; r < p->rec_slot.size(); r++) {
        cudaError_t e = cudaEventSynchronize(p->ev[2 * r + 1]);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, p->ev[2 * r], p->ev[2 * r + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "moe_profile_read");
        int s = p->rec_slot[r];
        if (s < n_slots) {
            total_ms[s] += ms;
            launches[s] += 1;
        }
    }
    p->rec_slot.clear();
    return MOE_OK;
}

int moe_get_device_status(moe_plan *p, int *status, void *stream) {
    if (!p || !status) return fail(MOE_EINVAL, "NULL argument");
    int32_t *words[2] = {nullptr, nullptr};
    int nw = 0;
    if (p->have_ws) words[nw++] = p->ws.status;
    if (p->noalloc_dev >= 0) {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "moe_get_device_status");
        void *base = nullptr;
        if (dev == p->noalloc_dev && noalloc_scratch_addr(dev, &base) == MOE_OK)
            words[nw++] = static_cast<int32_t *>(base);  // the static array's status word
    }
    if (!nw) return fail(MOE_ENOTREADY, "no workspace and no moe_forward_noalloc on the current device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < nw && e == cudaSuccess; i++) e = cudaMemcpyAsync(h[i], words[i], 16, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    for (int i = 0; i < nw && e == cudaSuccess; i++) e = cudaMemsetAsync(words[i], 0, 16, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_get_device_status");
    *status = 0;
    for (int i = 0; i < nw; i++)
        if (h[i][0]) {
            *status = h[i][0];
            return fail(MOE_EDEVICE, "device status %d (detail %d)%s", h[i][0], h[i][1],
                        words[i] == p->ws.status && p->have_ws ? "" : " in moe_forward_noalloc");
        }
    return MOE_OK;
}


int moe_cast_f32_to_bf16(const float *src, uint16_t *dst, size_t n, void *stream) {
    if (n == 0) return MOE_OK;
    if (!src || !dst) return fail(MOE_EINVAL, "NULL src or dst");
    if (!aligned16(src) || !aligned16(dst)) return fail(MOE_EINVAL, "src and dst must be 16-byte aligned");
    const char *sb = reinterpret_cast<const char *>(src), *db = reinterpret_cast<const char *>(dst);
    if (sb < db + n * 2 && db < sb + n * 4) return fail(MOE_EINVAL, "src and dst must not overlap");
    const cudaError_t e = launch_cast_bf16(src, dst, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_cast_f32_to_bf16");
}

int moe_mx_quantize_fp4(const uint16_t *x, size_t rows, size_t cols, uint8_t *codes, uint8_t *scales,
                        void *stream) {
    if (rows == 0) return MOE_OK;
    if (!x || !codes || !scales) return fail(MOE_EINVAL, "NULL x, codes or scales");
    if (cols == 0 || cols % 32 != 0) return fail(MOE_ESHAPE, "cols must be a positive multiple of 32 (got %zu)", cols);
    if (!aligned16(x) || !aligned16(codes)) return fail(MOE_EINVAL, "x and codes must be 16-byte aligned");
    if (rows > (SIZE_MAX / 2) / cols) return fail(MOE_EINVAL, "rows x cols overflows the address space");
    const size_t n = rows * cols;
    const char *xb = reinterpret_cast<const char *>(x), *cb = reinterpret_cast<const char *>(codes),
               *sb = reinterpret_cast<const char *>(scales);
    const size_t xn = n * 2, cn = n / 2, sn = n / 32;
    if ((xb < cb + cn && cb < xb + xn) || (xb < sb + sn && sb < xb + xn) || (cb < sb + sn && sb < cb + cn))
        return fail(MOE_EINVAL, "x, codes and scales must not overlap");
    const cudaError_t e = launch_mx_fp4_quantize(x, n / 32, codes, scales, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_mx_quantize_fp4");
}

int moe_forward_noalloc(moe_plan *p, const uint16_t *x, int tokens, float *out, int32_t *ids_out, void *stream) {
    if (!p) return fail(MOE_EINVAL, "NULL plan");
    if (tokens < 0) return fail(MOE_EINVAL, "tokens must be >= 0");
    if (tokens == 0) return MOE_OK;
    if (!x || !out) return fail(MOE_EINVAL, "NULL x or out");
    if (!p->have_w) return fail(MOE_ENOTREADY, "moe_load_weights has not been called");
    if (!aligned16(x) || !aligned16(out)) return fail(MOE_EINVAL, "x and out must be 16-byte aligned");
    if (tokens > kMaxTokens) return fail(MOE_ENOMEM, "moe_forward_noalloc: tokens %d > %d", tokens, kMaxTokens);
    const BlockParams &b = p->bp;
    const char *xb = reinterpret_cast<const char *>(x), *ob = reinterpret_cast<const char *>(out);
    if (xb < ob + (size_t)tokens * b.H * (p->out_bf16 ? 2 : 4) && ob < xb + (size_t)tokens * b.H * 2)
        return fail(MOE_EINVAL, "x and out must not alias");
    if (int rc0 = check_outputs(b, tokens, x, ids_out, nullptr, nullptr)) return rc0;
    const size_t need = carve(p, tokens, nullptr, nullptr);
    if (need > MOE_NOALLOC_SCRATCH_BYTES - MOE_NOALLOC_STATUS_BYTES)
        return fail(MOE_ENOMEM, "moe_forward_noalloc: %d tokens need %zu bytes of scratch, the static array holds %u",
                    tokens, need, MOE_NOALLOC_SCRATCH_BYTES - MOE_NOALLOC_STATUS_BYTES);
    {
        bool decode = false;
        int nt = 1, tile_rows = 0;
        if (int rc2 = choose_path(p, tokens, &decode, &nt, &tile_rows)) return rc2;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "moe_forward_noalloc: cudaGetDevice");
    void *base = nullptr;
    if (int rc = noalloc_scratch_addr(dev, &base)) return rc;
    Workspace ws;
    carve(p, tokens, static_cast<char *>(base) + MOE_NOALLOC_STATUS_BYTES, &ws);
    // the status word sits at the start of the array, where moe_get_device_status
    // finds it whatever the token count; like the workspace's, it is sticky
    // until read (a failure stays visible, later results are void until then)
    ws.status = static_cast<int32_t *>(base);
    p->noalloc_dev = dev;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents, and the routing kernel's
    // tickets (whose place depends on the token count) must start at zero
    e = cudaMemsetAsync(ws.tickets, 0, sizeof(uint32_t) * route_ticket_count(tokens), st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_forward_noalloc: clearing scratch");
    return enqueue_forward(p, ws, x, tokens, out, ids_out, nullptr, nullptr, st, [](int, bool) {});
}

}  // extern "C"
