// moe_cache.cu -- the expert cache: the expert matrices stay in a store the
// GPU can read but that need not be HBM (pinned host memory, read over the
// CPU-GPU link), and C of them at a time are kept in device slots.
//
// antirez ds4 (ds4.c) keeps an expert cache beside its expert profiler
// (`ds4_expert_profile_record`, `_cache_use`), and goosedump gpt_oss.rs
// streams expert bytes from storage through a lease cache (`ExpertStore`).
// Here the store is host memory, the cache is C device slots, and the choice
// of slots and the copies run on the device right after the routing, so a
// forward needs no host round trip and stays capturable in a CUDA graph.
//
// Policy, per forward: the experts the forward routes to are taken in
// ascending order; a resident one is a hit and its slot is stamped with the
// forward's index; a missing one takes the slot with the oldest stamp among
// the slots this forward has not stamped (empty slots carry stamp -1; the
// lowest slot index on a tie), evicting that slot's expert.  Every tile of the
// forward then names its expert's slot (the tile table's fourth field), and
// the missing experts' bytes are copied from the store into their slots
// before the GEMVs read them.  The shared expert is not cached (every token
// uses it): the plan keeps a device copy.
#include <climits>

#include "moe_common.cuh"

namespace {

__global__ void __launch_bounds__(32) moe_cache_assign_kernel(CacheTables c, BlockParams bp, Workspace ws) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the routing's counts and tiles
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x, E = bp.E, C = c.slots;
    const long long now = *c.fwd + 1;
    int hits = 0;
    // hits: stamp the resident experts this forward uses
    for (int e = lane; e < E; e += 32)
        if (ws.counts[e] > 0 && c.slot_of[e] >= 0) {
            c.stamp[c.slot_of[e]] = now;
            hits++;
        }
#pragma unroll
    for (int o = 16; o; o >>= 1) hits += __shfl_xor_sync(0xffffffffu, hits, o);
    __syncwarp();
    // misses, in ascending expert order: the least recently stamped slot not
    // stamped by this forward
    int n_miss = 0;
    bool full = false;
    for (int e0 = 0; e0 < E && !full; e0 += 32) {
        const int e = e0 + lane;
        unsigned need = __ballot_sync(0xffffffffu, e < E && ws.counts[e] > 0 && c.slot_of[e] < 0);
        while (need) {
            const int ee = e0 + __ffs(need) - 1;
            need &= need - 1;
            long long bs = LLONG_MAX;
            int bi = C;
            for (int s = lane; s < C; s += 32) {
                const long long st = c.stamp[s];
                if (st != now && (st < bs || (st == bs && s < bi))) {
                    bs = st;
                    bi = s;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const long long os = __shfl_xor_sync(0xffffffffu, bs, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (os < bs || (os == bs && oi < bi)) {
                    bs = os;
                    bi = oi;
                }
            }
            if (bi >= C) {  // more experts in this forward than slots (the host refuses such calls)
                if (lane == 0) set_device_error(ws.status, MOE_DEV_BAD_ROUTE, -3);
                full = true;
                break;
            }
            if (lane == 0) {
                const int old = c.expert_of[bi];
                if (old >= 0) c.slot_of[old] = -1;
                c.expert_of[bi] = ee;
                c.slot_of[ee] = bi;
                c.stamp[bi] = now;
                c.miss[n_miss] = make_int2(ee, bi);
            }
            n_miss++;
            __syncwarp();
        }
    }
    __syncwarp();
    // each tile names its expert's slot (the shared expert's tiles keep 0)
    const int nt = *ws.n_tiles;
    for (int i = lane; i < nt; i += 32) {
        const int e = ws.tiles[i].x;
        ws.tiles[i].w = e < E ? max(0, c.slot_of[e]) : 0;
    }
    if (lane == 0) {
        *c.n_miss = full ? 0 : n_miss;
        c.stats[0] += hits;
        c.stats[1] += n_miss;
        c.stats[2] += 1;
        *c.fwd = now;
    }
}

// The missing experts' matrices (codes, scales and biases of gate, up and
// down: kCacheArrays arrays, words[a] 16-byte words per expert each) from the
// store into their slots, as one flat range of words (every miss's arrays
// back to back); eight words per thread and round in flight.  The host keeps
// E x (words per expert) below 2^31, so the index math is 32-bit.
__global__ void __launch_bounds__(256) moe_cache_copy_kernel(CacheTables c, CacheArrays arr) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the slot assignment
    asm volatile("griddepcontrol.launch_dependents;");
    const int n = *c.n_miss;
    if (n == 0) return;
    unsigned W = 0;
#pragma unroll
    for (int a = 0; a < kCacheArrays; a++) W += (unsigned)arr.words[a];
    const unsigned total = (unsigned)n * W, stride = gridDim.x * blockDim.x;
    auto locate = [&](unsigned idx, const uint4 *&src, uint4 *&dst) {
        const unsigned j = idx / W;
        unsigned r = idx - j * W;
        int a = 0;
        while (a < kCacheArrays - 1 && r >= (unsigned)arr.words[a]) r -= (unsigned)arr.words[a++];
        const int2 m = c.miss[j];
        src = arr.src[a] + (size_t)m.x * arr.words[a] + r;
        dst = arr.dst[a] + (size_t)m.y * arr.words[a] + r;
    };
    constexpr int kIn = 8;
    for (unsigned base = blockIdx.x * blockDim.x + threadIdx.x; base < total; base += kIn * stride) {
        uint4 v[kIn];
        uint4 *d[kIn];
#pragma unroll
        for (int q = 0; q < kIn; q++) {
            const unsigned idx = base + q * stride;
            d[q] = nullptr;
            if (idx < total) {
                const uint4 *s;
                locate(idx, s, d[q]);
                v[q] = *s;
            }
        }
#pragma unroll
        for (int q = 0; q < kIn; q++)
            if (d[q]) *d[q] = v[q];
    }
}

}  // namespace

cudaError_t launch_cache_assign(const CacheTables &c, const BlockParams &bp, const Workspace &ws, cudaStream_t st) {
    return launch_pdl(moe_cache_assign_kernel, dim3(1), dim3(32), 0, st, c, bp, ws);
}

cudaError_t launch_cache_copy(const CacheTables &c, const CacheArrays &arr, cudaStream_t st) {
    int dev = 0, n_sm = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    return launch_pdl(moe_cache_copy_kernel, dim3(n_sm), dim3(256), 0, st, c, arr);
}
