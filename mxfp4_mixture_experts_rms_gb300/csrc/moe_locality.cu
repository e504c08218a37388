// moe_locality.cu -- expert-locality statistics of the routing, recorded on
// the device after each forward: antirez ds4, ds4.c, the Metal expert
// locality profiler (`ds4_expert_profile_record`,
// `ds4_expert_profile_cache_use`), whose per-layer selection histogram is also
// goosedump gpt_oss.rs `ExpertRouteProfile`.
//
// Per layer: selections and route weight per expert; the overlap of the
// expert sets of tokens at consecutive positions; and, for each cache
// capacity, the hits a least-recently-used cache of that many experts would
// see.  The pages keep one most-recently-used list per capacity and move each
// used expert to its front.  Here one pass serves every capacity at once: the
// list of capacity c holds exactly the c experts used most recently, so an
// access hits it iff fewer than c distinct experts were used since the
// expert's own last use.  Each expert keeps the time of its last use (a
// per-layer counter of accesses); that number is the count of experts whose
// last use is later.  The accesses of a layer are taken in the pages' order
// (token, then slot) by one warp with integer work only; the weights of the
// hits are then summed by the warp's lanes (a fixed order, not the pages'
// sequential one: the same sums up to rounding).
#include "moe_common.cuh"
#include "../../include/moe.h"

#include <cstdlib>
#include <cstring>

namespace {

constexpr int kLocMaxCaps = 16;

// Device state of one profiler (one allocation, carved in this order).
struct LocState {
    unsigned long long *hist;       // [L][E] selections
    double *whist;                  // [L][E] route weight
    unsigned long long *records;    // [L] recorded tokens
    unsigned long long *adj;        // [L][K + 1] adjacent pairs by intersection size
    unsigned long long *last_use;   // [L][E] access time of the last use (0: never)
    unsigned long long *clock;      // [L] accesses so far
    long long *prev_pos;            // [L] position of the previous recorded token (none: -2^62)
    int *prev_sel;                  // [L][K] its selected experts
    unsigned long long *hits;       // [C][L]
    double *whits;                  // [C][L]
};

struct LocDims {
    int L, E, K, C;
    int caps[kLocMaxCaps];
};

size_t loc_carve(const LocDims &d, unsigned char *base, LocState *s) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        unsigned char *p = base ? base + off : nullptr;
        off = (off + bytes + 255) & ~(size_t)255;
        return p;
    };
    const size_t L = d.L, E = d.E, K = d.K, C = d.C;
    LocState t;
    t.hist = reinterpret_cast<unsigned long long *>(take(L * E * 8));
    t.whist = reinterpret_cast<double *>(take(L * E * 8));
    t.records = reinterpret_cast<unsigned long long *>(take(L * 8));
    t.adj = reinterpret_cast<unsigned long long *>(take(L * (K + 1) * 8));
    t.last_use = reinterpret_cast<unsigned long long *>(take(L * E * 8));
    t.clock = reinterpret_cast<unsigned long long *>(take(L * 8));
    t.prev_pos = reinterpret_cast<long long *>(take(L * 8));
    t.prev_sel = reinterpret_cast<int *>(take(L * K * 4));
    t.hits = reinterpret_cast<unsigned long long *>(take(C * L * 8));
    t.whits = reinterpret_cast<double *>(take(C * L * 8));
    if (s) *s = t;
    return off;
}

constexpr int kLocThreads = 256;
constexpr int kLocChunk = 1024;  // selections staged in shared memory at a time

// Adjacent tokens: token t against t - 1 (token 0 against the layer's
// previous record if that sat at first_pos - 1), threads i0, i0 + step, ...
__device__ void adjacent(const LocState &s, const LocDims &d, int layer, const int32_t *ids, int T,
                         long long first_pos, int i0, int step) {
    const int K = d.K;
    for (int t = i0; t < T; t += step) {
        const int *prev;
        if (t == 0) {
            if (s.prev_pos[layer] != first_pos - 1) continue;
            prev = s.prev_sel + (size_t)layer * K;
        } else {
            prev = ids + (size_t)(t - 1) * K;
        }
        const int *cur = ids + (size_t)t * K;
        int inter = 0;
        for (int a = 0; a < K; a++) {
            const int pa = prev[a];
            for (int b = 0; b < K; b++)
                if (pa == cur[b]) {
                    inter++;
                    break;
                }
        }
        atomicAdd(s.adj + (size_t)layer * (K + 1) + inter, 1ull);
    }
}

// One launch records T tokens of one layer at positions first_pos + t.
// Warp 0: the cache pass (sequential in access order).  The other warps: the
// histograms (atomics) and the adjacent-token overlaps.
__global__ void __launch_bounds__(kLocThreads) moe_locality_kernel(LocState s, LocDims d, int layer, const int32_t *ids,
                                                                 const float *w, int T, long long first_pos) {
    __shared__ int s_ids[kLocChunk];
    __shared__ float s_w[kLocChunk];
    __shared__ int s_dist[kLocChunk];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = d.E, K = d.K, n = T * K;
    if (warp == 0) {
        // expert e's last use lives in lane e % 32, register slot e / 32
        constexpr int kSlots = MOE_MAX_EXPERTS / 32;
        unsigned long long *last = s.last_use + (size_t)layer * E;
        unsigned long long lr[kSlots];
#pragma unroll
        for (int k = 0; k < kSlots; k++) lr[k] = 32 * k + lane < E ? last[32 * k + lane] : 0ull;
        unsigned long long clk = s.clock[layer];
        unsigned long long hits[kLocMaxCaps];  // registers: every index below is a constant
        double whits[kLocMaxCaps];
#pragma unroll
        for (int c = 0; c < kLocMaxCaps; c++) {
            hits[c] = 0;
            whits[c] = 0.0;
        }
        for (int i0 = 0; i0 < n; i0 += kLocChunk) {
            // the next chunk of selections into shared memory (coalesced)
            const int m = min(kLocChunk, n - i0);
            for (int i = lane; i < m; i += 32) {
                s_ids[i] = ids[i0 + i];
                s_w[i] = w[i0 + i];
            }
            __syncwarp();
            // in access order: each selection's count of experts used since the
            // expert's last use (a hit for every larger capacity; never used
            // before or skipped: a hit for none), integer work only, in registers
            for (int i = 0; i < m; i++) {
                const int e = s_ids[i];
                int dist = 0x7fffffff;
                if (e >= 0 && e < E) {
                    const int slot = e >> 5, owner = e & 31;
                    unsigned long long mine = 0;
#pragma unroll
                    for (int k = 0; k < kSlots; k++)
                        if (k == slot) mine = lr[k];
                    const unsigned long long lu = __shfl_sync(0xffffffffu, mine, owner);
                    if (lu) {
                        int later = 0;
#pragma unroll
                        for (int k = 0; k < kSlots; k++)
                            if (32 * k < E) later += __popc(__ballot_sync(0xffffffffu, lr[k] > lu));
                        dist = later;
                    }
                    ++clk;
                    if (lane == owner) {
#pragma unroll
                        for (int k = 0; k < kSlots; k++)
                            if (k == slot) lr[k] = clk;
                    }
                }
                if (lane == 0) s_dist[i] = dist;
            }
            __syncwarp();
            // hits and hit weights per capacity, the lanes over the chunk's selections
#pragma unroll
            for (int c = 0; c < kLocMaxCaps; c++) {
                if (c >= d.C) break;
                unsigned long long h = 0;
                double wsum = 0.0;
                for (int i = lane; i < m; i += 32)
                    if (s_dist[i] < d.caps[c]) {
                        h++;
                        wsum += (double)s_w[i];
                    }
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    h += __shfl_xor_sync(0xffffffffu, h, o);
                    wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
                }
                hits[c] += h;
                whits[c] += wsum;
            }
            __syncwarp();
        }
#pragma unroll
        for (int k = 0; k < kSlots; k++)
            if (32 * k + lane < E) last[32 * k + lane] = lr[k];
        if (lane == 0) {
            s.clock[layer] = clk;
#pragma unroll
            for (int c = 0; c < kLocMaxCaps; c++)
                if (c < d.C) {
                    s.hits[(size_t)c * d.L + layer] += hits[c];
                    s.whits[(size_t)c * d.L + layer] += whits[c];
                }
        }
    } else {
        // selections and weights per expert
        for (int i = tid - 32; i < n; i += kLocThreads - 32) {
            const int e = ids[i];
            if (e < 0 || e >= E) continue;
            atomicAdd(s.hist + (size_t)layer * E + e, 1ull);
            atomicAdd(s.whist + (size_t)layer * E + e, (double)w[i]);
        }
        adjacent(s, d, layer, ids, T, first_pos, tid - 32, kLocThreads - 32);
    }
    // the layer's previous token becomes the batch's last one, once every
    // comparison above has read the old one
    __syncthreads();
    for (int a = tid; a < K; a += kLocThreads) s.prev_sel[(size_t)layer * K + a] = ids[(size_t)(T - 1) * K + a];
    if (tid == 0) {
        s.prev_pos[layer] = first_pos + T - 1;
        s.records[layer] += (unsigned long long)T;
    }
}

}  // namespace

struct moe_locality {
    LocDims d;
    unsigned char *dev = nullptr;
    size_t bytes = 0;
    LocState s;
};

cudaError_t locality_enqueue(moe_locality *p, int layer, const int32_t *ids, const float *w, int T,
                             long long first_pos, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    moe_locality_kernel<<<1, kLocThreads, 0, st>>>(p->s, p->d, layer, ids, w, T, first_pos);
    return cudaGetLastError();
}

extern "C" {

moe_locality *moe_locality_create(int n_layers, int n_experts, int top_k, const int *caps, int n_caps) {
    if (n_layers < 1 || n_layers > 4096 || n_experts < 1 || n_experts > MOE_MAX_EXPERTS || top_k < 1 ||
        top_k > 8 || top_k > n_experts || n_caps < 0 || n_caps > kLocMaxCaps || (n_caps && !caps)) {
        moe_set_error("moe_locality_create: bad arguments (1..4096 layers, 1..%d experts, 1..min(8, experts) "
                      "slots, 0..%d capacities)", MOE_MAX_EXPERTS, kLocMaxCaps);
        return nullptr;
    }
    LocDims d;
    d.L = n_layers;
    d.E = n_experts;
    d.K = top_k;
    d.C = 0;
    for (int i = 0; i < n_caps; i++)  // as the pages do, capacities outside 1..E are left out
        if (caps[i] >= 1 && caps[i] <= n_experts) d.caps[d.C++] = caps[i];
    moe_locality *p = new moe_locality;
    p->d = d;
    p->bytes = loc_carve(d, nullptr, nullptr);
    cudaError_t e = cudaMalloc(&p->dev, p->bytes);
    if (e != cudaSuccess) {
        moe_set_error("moe_locality_create: cudaMalloc: %s", cudaGetErrorString(e));
        delete p;
        return nullptr;
    }
    loc_carve(d, p->dev, &p->s);
    if (moe_locality_reset(p, nullptr) != MOE_OK || cudaStreamSynchronize(0) != cudaSuccess) {
        cudaFree(p->dev);
        delete p;
        return nullptr;
    }
    return p;
}

int moe_locality_reset(moe_locality *p, void *stream) {
    if (!p) return moe_fail_status(MOE_EINVAL, "NULL profiler");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(p->dev, 0, p->bytes, st);
    // no previous token: a position no first_pos - 1 can equal
    const long long none = -(1ll << 62);
    for (int l = 0; l < p->d.L && e == cudaSuccess; l++)
        e = cudaMemcpyAsync(p->s.prev_pos + l, &none, sizeof(none), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? MOE_OK : moe_fail_status(MOE_ECUDA, "moe_locality_reset: %s", cudaGetErrorString(e));
}

int moe_locality_record(moe_locality *p, int layer, const int32_t *ids, const float *route_w, int tokens,
                        long long first_pos, void *stream) {
    if (!p) return moe_fail_status(MOE_EINVAL, "NULL profiler");
    if (layer < 0 || layer >= p->d.L) return moe_fail_status(MOE_EINVAL, "layer %d out of range", layer);
    if (tokens < 0) return moe_fail_status(MOE_EINVAL, "tokens must be >= 0");
    if (tokens == 0) return MOE_OK;
    if (!ids || !route_w) return moe_fail_status(MOE_EINVAL, "NULL ids or route weights");
    if (reinterpret_cast<uintptr_t>(ids) % 4 || reinterpret_cast<uintptr_t>(route_w) % 4)
        return moe_fail_status(MOE_EINVAL, "ids and route weights must be 4-byte aligned");
    const cudaError_t e = locality_enqueue(p, layer, ids, route_w, tokens, first_pos, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : moe_fail_status(MOE_ECUDA, "moe_locality_record: %s", cudaGetErrorString(e));
}

int moe_locality_read(const moe_locality *p, moe_locality_stats *out) {
    if (!p || !out) return moe_fail_status(MOE_EINVAL, "NULL argument");
    const LocDims &d = p->d;
    unsigned char *h = static_cast<unsigned char *>(malloc(p->bytes));
    if (!h) return moe_fail_status(MOE_ENOMEM, "moe_locality_read: host buffer");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(h, p->dev, p->bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        free(h);
        return moe_fail_status(MOE_ECUDA, "moe_locality_read: %s", cudaGetErrorString(e));
    }
    LocState s;
    loc_carve(d, h, &s);
    const size_t LE = (size_t)d.L * d.E;
    if (out->hist) memcpy(out->hist, s.hist, LE * 8);
    if (out->weight_hist) memcpy(out->weight_hist, s.whist, LE * 8);
    if (out->layer_records) memcpy(out->layer_records, s.records, (size_t)d.L * 8);
    for (int l = 0; l < d.L; l++) {
        unsigned long long pairs = 0;
        double ov = 0.0, jac = 0.0;
        for (int i = 0; i <= d.K; i++) {
            const unsigned long long c = s.adj[(size_t)l * (d.K + 1) + i];
            pairs += c;
            ov += (double)c * ((double)i / (double)d.K);
            jac += (double)c * ((double)i / (double)(2 * d.K - i));
        }
        if (out->adjacent_pairs) out->adjacent_pairs[l] = pairs;
        if (out->overlap_sum) out->overlap_sum[l] = ov;
        if (out->jaccard_sum) out->jaccard_sum[l] = jac;
    }
    if (out->cache_hits) memcpy(out->cache_hits, s.hits, (size_t)d.C * d.L * 8);
    if (out->cache_weight_hits) memcpy(out->cache_weight_hits, s.whits, (size_t)d.C * d.L * 8);
    if (out->caps)
        for (int c = 0; c < d.C; c++) out->caps[c] = d.caps[c];
    out->n_caps = d.C;
    free(h);
    return MOE_OK;
}

void moe_locality_destroy(moe_locality *p) {
    if (!p) return;
    cudaFree(p->dev);
    delete p;
}

}  // extern "C"
