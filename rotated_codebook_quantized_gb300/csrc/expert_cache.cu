// Expert streaming: a bank of experts larger than the device's budget stays in
// host memory, and the experts a step routes to are copied into a device cache
// of slots managed least-recently-used.
//
// "How it works", "Expert streaming": for a Mixture-of-Experts model bigger
// than memory only the shared parts stay resident; the experts each token
// routes to are read (in parallel, with an LRU cache) and the result is
// bit-identical to running it in memory.  "Running a 1T-Parameter Model on a
// Laptop": load_experts(expert_ids) reads only the routed experts.  On GB300
// the bank lives in pinned host memory and a miss is two host-to-device copies
// (code words and scales) into the slot the LRU gives up; the gather kernels
// then read the slot bank with the ids remapped to slots.
//
// Host code only: the cache object holds the bookkeeping (slot contents and
// last use); the slot buffers on the device and the pinned bank belong to the
// caller.
#include <string.h>

#include <new>
#include <vector>

#include "common.cuh"

struct tq_expert_cache {
    tq_qweight_t host;              // the bank (host pointers)
    uint32_t* dev_codes;            // [slots][rows][row_stride_words]
    uint16_t* dev_scales;           // [slots][rows][cols/group]
    int slots;
    std::vector<int> slot_expert;   // expert held by each slot, -1 if empty
    std::vector<int64_t> last_use;  // step of each slot's last use (0: never)
    std::vector<int> expert_slot;   // slot of each expert, -1 if not cached
    std::vector<int64_t> seen;      // step in which each expert was last looked up
    bool kernel_copy = false;       // the bank is pinned, mapped and 16-byte aligned: copied by a kernel
    int64_t step = 0;
    int64_t hits = 0, misses = 0, bytes = 0;
};

using namespace tq;

namespace {

size_t expert_code_bytes(const tq_qweight_t& w) { return (size_t)w.rows * w.row_stride_words * 4; }
size_t expert_scale_bytes(const tq_qweight_t& w) { return (size_t)w.rows * (w.cols / w.group) * 2; }

// One launch copies every missing expert: the threads of the grid walk each segment in turn with
// 16-byte loads straight from the pinned bank (mapped into the device's address space, read over
// the CPU-GPU link), four loads in flight per thread.
constexpr int kMaxSegs = 64;
struct CopySegs {
    const uint4* src[kMaxSegs];
    uint4* dst[kMaxSegs];
    int64_t n16[kMaxSegs];  // 16-byte pieces
    int nseg;
};

__global__ void __launch_bounds__(256) stream_copy_kernel(const CopySegs cs) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int sg = 0; sg < cs.nseg; ++sg) {
        const uint4* __restrict__ src = cs.src[sg];
        uint4* __restrict__ dst = cs.dst[sg];
        const int64_t n = cs.n16[sg];
        int64_t i = t;
        for (; i + 3 * stride < n; i += 4 * stride) {
            const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
            dst[i] = a;
            dst[i + stride] = b;
            dst[i + 2 * stride] = c;
            dst[i + 3 * stride] = d;
        }
        for (; i < n; i += stride) dst[i] = src[i];
    }
}

bool device_readable(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

// LRU bookkeeping of one step: the slot of every id in slots_out[], and miss[i] = 1 for the
// first occurrence of each expert that has to be copied.  Hits and misses count distinct
// experts of the step.  An expert used in this step is never evicted by another of it.
tq_status plan(tq_expert_cache* c, const int32_t* ids, int32_t n, int32_t* slots_out, uint8_t* miss) {
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= c->host.experts) return TQ_ERR_INVALID;
    const int64_t now = ++c->step;
    int distinct_missing = 0;
    for (int i = 0; i < n; ++i) {
        const int e = ids[i];
        if (c->seen[e] == now) continue;
        c->seen[e] = now;
        const int s = c->expert_slot[e];
        if (s >= 0)
            c->last_use[s] = now;  // hits first, so that no miss of this step takes their slots
        else
            ++distinct_missing;
    }
    int free_slots = 0;
    for (int k = 0; k < c->slots; ++k) free_slots += c->last_use[k] != now;
    if (distinct_missing > free_slots) return TQ_ERR_INVALID;  // more distinct experts than slots
    for (int i = 0; i < n; ++i) {
        const int e = ids[i];
        miss[i] = 0;
        const int s = c->expert_slot[e];
        if (s >= 0) {
            if (c->seen[e] == now) ++c->hits;  // first occurrence: mark the expert counted
            c->seen[e] = now - 1;
            slots_out[i] = s;
            continue;
        }
        // victim: an empty slot, else the least recently used slot not used in this step
        int v = -1;
        for (int k = 0; k < c->slots; ++k) {
            if (c->last_use[k] == now) continue;
            if (c->slot_expert[k] < 0) {
                v = k;
                break;
            }
            if (v < 0 || c->last_use[k] < c->last_use[v]) v = k;
        }
        if (c->slot_expert[v] >= 0) c->expert_slot[c->slot_expert[v]] = -1;
        c->slot_expert[v] = e;
        c->expert_slot[e] = v;
        c->last_use[v] = now;
        c->seen[e] = now - 1;
        slots_out[i] = v;
        miss[i] = 1;
        ++c->misses;
    }
    return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_expert_cache_create(const tq_qweight_t* host_bank, int32_t slots, uint32_t* dev_codes,
                                            uint16_t* dev_scales, tq_expert_cache** out) {
    if (!host_bank || !out || slots <= 0 || host_bank->experts <= 0 || host_bank->rows <= 0 || host_bank->cols <= 0)
        return TQ_ERR_INVALID;
    if (!(host_bank->group == 16 || host_bank->group == 32 || host_bank->group == 64 || host_bank->group == 128) ||
        host_bank->cols % host_bank->group || host_bank->row_stride_words < tq_row_words(host_bank->cb.levels,
                                                                                         host_bank->cols))
        return TQ_ERR_INVALID;
    if (host_bank->experts > 1 &&
        (host_bank->expert_stride_words != (int64_t)host_bank->rows * host_bank->row_stride_words ||
         host_bank->expert_stride_scales != (int64_t)host_bank->rows * (host_bank->cols / host_bank->group)))
        return TQ_ERR_UNSUPPORTED;  // experts stored back to back (one copy per tensor per expert)
    tq_expert_cache* c = new (std::nothrow) tq_expert_cache();
    if (!c) return TQ_ERR_INVALID;
    c->host = *host_bank;
    c->dev_codes = dev_codes;
    c->dev_scales = dev_scales;
    c->slots = slots;
    c->slot_expert.assign(slots, -1);
    c->last_use.assign(slots, 0);
    c->expert_slot.assign(host_bank->experts, -1);
    c->seen.assign(host_bank->experts, 0);
    const size_t cbytes = expert_code_bytes(c->host), sbytes = expert_scale_bytes(c->host);
    c->kernel_copy = cbytes % 16 == 0 && sbytes % 16 == 0 && aligned(c->host.codes, 16) &&
                     aligned(c->host.scales, 16) && aligned(dev_codes, 16) && aligned(dev_scales, 16) &&
                     device_readable(c->host.codes) && device_readable(c->host.scales);
    *out = c;
    return TQ_OK;
}

extern "C" void tq_expert_cache_destroy(tq_expert_cache* c) { delete c; }

extern "C" tq_status tq_expert_cache_plan(tq_expert_cache* c, const int32_t* ids, int32_t n, int32_t* slots,
                                          uint8_t* miss) {
    if (!c || n < 0 || (n > 0 && (!ids || !slots || !miss))) return TQ_ERR_INVALID;
    return plan(c, ids, n, slots, miss);
}

extern "C" tq_status tq_expert_cache_map(tq_expert_cache* c, const int32_t* ids, int32_t n, int32_t* slots,
                                         void* stream) {
    if (!c || n < 0 || (n > 0 && (!ids || !slots))) return TQ_ERR_INVALID;
    if (!c->dev_codes || !c->dev_scales || !c->host.codes || !c->host.scales) return TQ_ERR_INVALID;
    std::vector<uint8_t> miss(n);
    const tq_status s = plan(c, ids, n, slots, miss.data());
    if (s != TQ_OK) return s;
    const size_t cb = expert_code_bytes(c->host), sb = expert_scale_bytes(c->host);
    cudaStream_t st = as_stream(stream);
    if (c->kernel_copy) {
        CopySegs segs{};
        auto flush = [&]() -> tq_status {
            if (segs.nseg == 0) return TQ_OK;
            int sms = 0, dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            stream_copy_kernel<<<4 * (sms > 0 ? sms : 152), 256, 0, st>>>(segs);
            segs.nseg = 0;
            return launch_status();
        };
        for (int i = 0; i < n; ++i) {
            if (!miss[i]) continue;
            const int e = ids[i], v = slots[i];
            if (segs.nseg + 2 > kMaxSegs) {
                const tq_status fs = flush();
                if (fs != TQ_OK) return fs;
            }
            segs.src[segs.nseg] = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(c->host.codes) + (size_t)e * cb);
            segs.dst[segs.nseg] = reinterpret_cast<uint4*>(reinterpret_cast<char*>(c->dev_codes) + (size_t)v * cb);
            segs.n16[segs.nseg++] = (int64_t)(cb / 16);
            segs.src[segs.nseg] = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(c->host.scales) + (size_t)e * sb);
            segs.dst[segs.nseg] = reinterpret_cast<uint4*>(reinterpret_cast<char*>(c->dev_scales) + (size_t)v * sb);
            segs.n16[segs.nseg++] = (int64_t)(sb / 16);
            c->bytes += (int64_t)(cb + sb);
        }
        return flush();
    }
    for (int i = 0; i < n; ++i) {
        if (!miss[i]) continue;
        const int e = ids[i], v = slots[i];
        const char* hc = reinterpret_cast<const char*>(c->host.codes) + (size_t)e * cb;
        const char* hs = reinterpret_cast<const char*>(c->host.scales) + (size_t)e * sb;
        if (cudaMemcpyAsync(reinterpret_cast<char*>(c->dev_codes) + (size_t)v * cb, hc, cb, cudaMemcpyHostToDevice,
                            st) != cudaSuccess ||
            cudaMemcpyAsync(reinterpret_cast<char*>(c->dev_scales) + (size_t)v * sb, hs, sb, cudaMemcpyHostToDevice,
                            st) != cudaSuccess)
            return TQ_ERR_CUDA;
        c->bytes += (int64_t)(cb + sb);
    }
    return TQ_OK;
}

extern "C" tq_status tq_expert_cache_stats(const tq_expert_cache* c, int64_t* hits, int64_t* misses,
                                           int64_t* bytes_copied) {
    if (!c) return TQ_ERR_INVALID;
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (bytes_copied) *bytes_copied = c->bytes;
    return TQ_OK;
}
