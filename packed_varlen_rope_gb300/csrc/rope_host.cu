// Host-buffer streaming for packed QK-RoPE: Q and K live in (pinned) host memory; the
// library walks the pack in chunks of tokens through a device staging workspace,
// overlapping the host-to-device copy of chunk i+1, the rotation of chunk i and the
// device-to-host copy of chunk i-1 on three streams.  Each chunk is rotated by the
// same kernel as rope_qk_apply with its global token offset (or its slice of the
// position ids), so the results are those of one rotation of the whole pack.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rope_qk.h"

// rope_qk_apply with plain (not programmatically overlapped) launches (rope_qk.cu).
int rope_qk_apply_plain_launch(const rope_qk_desc *desc, void *stream);
// rope_qk_apply's checks that do not depend on where Q and K live (rope_qk.cu).
int rope_qk_check_pack(const rope_qk_desc *desc);

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 2;

// Streams and events of the pipeline, created once per device on first use and kept
// for the life of the process.
struct DeviceQueues {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t loaded[kSlots] = {}, rotated[kSlots] = {}, drained[kSlots] = {};
};

std::mutex g_mutex;
DeviceQueues g_queues[kMaxDevices];

int queues_for_current_device(DeviceQueues **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ROPE_ERR_LAUNCH;
    DeviceQueues &q = g_queues[dev];
    if (!q.ready) {
        const unsigned ev = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&q.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&q.d2h, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&q.entry, ev) != cudaSuccess)
            return ROPE_ERR_LAUNCH;
        for (int s = 0; s < kSlots; ++s)
            if (cudaEventCreateWithFlags(&q.loaded[s], ev) != cudaSuccess ||
                cudaEventCreateWithFlags(&q.rotated[s], ev) != cudaSuccess ||
                cudaEventCreateWithFlags(&q.drained[s], ev) != cudaSuccess)
                return ROPE_ERR_LAUNCH;
        q.ready = true;
    }
    *out = &q;
    return ROPE_OK;
}

bool contiguous(const void *p, int64_t ts, int64_t hs, int32_t heads, int32_t d)
{
    return p == nullptr || (hs == d && ts == static_cast<int64_t>(heads) * d);
}

// Everything a host-buffer call can be rejected for, checked on the whole pack before
// the first copy: the checks of rope_qk_apply that do not depend on where Q and K live
// (sizes, flags, theta and scale, positions, segments, the cache), the host buffers'
// layout, and the cache's device.  Every chunk's rotation then takes a descriptor that
// passes rope_qk_apply's checks (its views are slices of the staging memory, its
// positions a slice of the pack's), so no error other than one of the CUDA runtime can
// come after a copy.  Returns ROPE_OK for a call with work to do.
int check_host_call(const rope_qk_desc *dp)
{
    int rc = rope_qk_check_pack(dp);
    if (rc != ROPE_OK) return rc;
    const rope_qk_desc &p = *dp;
    if (p.total_tokens == 0) return ROPE_OK;
    if (p.q == nullptr || p.k == nullptr) return ROPE_ERR_NULL;
    if ((p.q_out == nullptr) != (p.k_out == nullptr)) return ROPE_ERR_NULL;
    const int32_t d = p.head_dim;
    if (!contiguous(p.q, p.q_stride_token, p.q_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k, p.k_stride_token, p.k_stride_head, p.n_kv_heads, d) ||
        !contiguous(p.q_out, p.q_out_stride_token, p.q_out_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k_out, p.k_out_stride_token, p.k_out_stride_head, p.n_kv_heads, d))
        return ROPE_ERR_SHAPE;
    const rope_cos_sin_cache *c = p.cos_sin_cache;
    if (c != nullptr && c->rows > 0) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return ROPE_ERR_LAUNCH;
        if (dev != c->device) return ROPE_ERR_CACHE;
    }
    return ROPE_OK;
}

// The position ids of rows [t0, ...) of a chunk: int32 or, with the flag, int64 values.
const int32_t *ids_from(const rope_qk_desc &p, int64_t t0)
{
    if ((p.flags & ROPE_FLAG_POSITION_IDS_INT64) != 0)
        return reinterpret_cast<const int32_t *>(reinterpret_cast<const int64_t *>(p.position_ids) + t0);
    return p.position_ids + t0;
}

// Descriptor of the rotation of rows [t0, t0 + n) of the pack, staged in place at dq
// (Q rows) and dk (K rows): the pack's descriptor with contiguous device views, its
// position ids, token offset or segment list moved to the chunk's first row.  `segs`
// receives the chunk's segments (the pack's, cut to the chunk and re-based).
rope_qk_desc chunk_desc(const rope_qk_desc &p, int64_t t0, int64_t n, void *dq, void *dk, rope_qk_segment *segs)
{
    rope_qk_desc cd = p;
    const int64_t d = p.head_dim;
    cd.q = dq;
    cd.k = dk;
    cd.q_stride_token = p.n_q_heads * d;
    cd.q_stride_head = d;
    cd.k_stride_token = p.n_kv_heads * d;
    cd.k_stride_head = d;
    cd.q_out = nullptr;
    cd.k_out = nullptr;
    cd.total_tokens = n;
    if (p.position_ids != nullptr) {
        cd.position_ids = ids_from(p, t0);
    } else if (p.n_segments == 0) {
        cd.token_offset = p.token_offset + t0;
    } else {
        int m = 0;
        for (int i = 0; i < p.n_segments; ++i) {
            const int64_t s0 = p.segments[i].row_start;
            const int64_t s1 = i + 1 < p.n_segments ? p.segments[i + 1].row_start : p.total_tokens;
            const int64_t lo = std::max(s0, t0), hi = std::min(s1, t0 + n);
            if (lo >= hi) continue;
            segs[m].row_start = lo - t0;
            segs[m].token_start = p.segments[i].token_start + (lo - s0);
            ++m;
        }
        cd.segments = segs;
        cd.n_segments = m;
    }
    return cd;
}

}  // namespace

// Shared by rope_qk_host and its static-workspace variant: stream the pack through
// `workspace` (device, workspace_bytes) on `stream`.
int rope_qk_host_impl(const rope_qk_desc *dp, void *workspace, int64_t workspace_bytes, void *stream)
{
    int rc = check_host_call(dp);
    if (rc != ROPE_OK) return rc;
    const rope_qk_desc &p = *dp;
    const int64_t T = p.total_tokens;
    if (workspace_bytes < 0) return ROPE_ERR_SHAPE;
    if (T == 0) return ROPE_OK;
    if (workspace == nullptr) return ROPE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ROPE_ERR_ALIGN;

    // chunk geometry: two slots, each holding the Q and K rows of `chunk` tokens
    const int32_t d = p.head_dim;
    const int64_t q_row = static_cast<int64_t>(p.n_q_heads) * d * 2;
    const int64_t k_row = static_cast<int64_t>(p.n_kv_heads) * d * 2;
    const int64_t per_token = q_row + k_row;
    int64_t chunk = workspace_bytes / (kSlots * per_token);
    chunk -= chunk % 8;                       // keep every slot's K part 16-byte aligned
    if (chunk < 8) return ROPE_ERR_UNSUPPORTED;
    if (chunk > T) chunk = T;
    if (chunk > (int64_t(1) << 24)) chunk = int64_t(1) << 24;
    const int64_t slot_bytes = ((chunk * per_token) + 255) / 256 * 256;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceQueues *qs = nullptr;
    rc = queues_for_current_device(&qs);
    if (rc != ROPE_OK) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // After a failure of the CUDA runtime the caller's stream still waits for every copy
    // already queued, so that freeing or reusing the workspace or the host buffers after
    // the error is ordered after them.
    auto join = [&]() {
        if (cudaEventRecord(qs->loaded[0], qs->h2d) == cudaSuccess) cudaStreamWaitEvent(s, qs->loaded[0], 0);
        if (cudaEventRecord(qs->drained[0], qs->d2h) == cudaSuccess) cudaStreamWaitEvent(s, qs->drained[0], 0);
    };
    bool ok = cudaEventRecord(qs->entry, s) == cudaSuccess &&
              cudaStreamWaitEvent(qs->h2d, qs->entry, 0) == cudaSuccess &&
              cudaStreamWaitEvent(qs->d2h, qs->entry, 0) == cudaSuccess;

    const int64_t n_chunks = (T + chunk - 1) / chunk;
    char *const q_host = static_cast<char *>(p.q);
    char *const k_host = static_cast<char *>(p.k);
    char *const qo_host = static_cast<char *>(p.q_out != nullptr ? p.q_out : p.q);
    char *const ko_host = static_cast<char *>(p.k_out != nullptr ? p.k_out : p.k);
    for (int64_t c = 0; ok && c < n_chunks; ++c) {
        const int slot = static_cast<int>(c % kSlots);
        const int64_t t0 = c * chunk;
        const int64_t n = (T - t0) < chunk ? (T - t0) : chunk;
        char *const dq = static_cast<char *>(workspace) + slot * slot_bytes;
        char *const dk = dq + chunk * q_row;
        // 1. host -> device, once the slot's previous contents have been copied out
        if (c >= kSlots) ok = ok && cudaStreamWaitEvent(qs->h2d, qs->drained[slot], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(dq, q_host + t0 * q_row, n * q_row, cudaMemcpyHostToDevice, qs->h2d) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(dk, k_host + t0 * k_row, n * k_row, cudaMemcpyHostToDevice, qs->h2d) == cudaSuccess;
        ok = ok && cudaEventRecord(qs->loaded[slot], qs->h2d) == cudaSuccess;
        // 2. rotate the chunk in place in the slot, on the caller's stream
        ok = ok && cudaStreamWaitEvent(s, qs->loaded[slot], 0) == cudaSuccess;
        if (!ok) break;
        rope_qk_segment segs[ROPE_MAX_SEGMENTS];
        const rope_qk_desc cd = chunk_desc(p, t0, n, dq, dk, segs);
        rc = rope_qk_apply_plain_launch(&cd, stream);
        if (rc != ROPE_OK) {
            join();
            return rc;
        }
        ok = cudaEventRecord(qs->rotated[slot], s) == cudaSuccess;
        // 3. device -> host
        ok = ok && cudaStreamWaitEvent(qs->d2h, qs->rotated[slot], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(qo_host + t0 * q_row, dq, n * q_row, cudaMemcpyDeviceToHost, qs->d2h) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(ko_host + t0 * k_row, dk, n * k_row, cudaMemcpyDeviceToHost, qs->d2h) == cudaSuccess;
        ok = ok && cudaEventRecord(qs->drained[slot], qs->d2h) == cudaSuccess;
    }
    // the caller's stream continues only after the last copies to the host
    for (int slot = 0; ok && slot < kSlots && slot < n_chunks; ++slot)
        ok = cudaStreamWaitEvent(s, qs->drained[slot], 0) == cudaSuccess;
    if (!ok) join();
    return ok ? ROPE_OK : ROPE_ERR_LAUNCH;
}

extern "C" int rope_qk_host(const rope_qk_desc *desc, void *workspace, int64_t workspace_bytes, void *stream)
{
    return rope_qk_host_impl(desc, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- allocation-free variant
//
// Staging memory that needs no allocation call: a file-scope device array.  Every GPU on
// which this library's device code is loaded keeps these 32 MiB until the process
// exits.  Host code must not use the array's name as a device address (on the host it
// is only a stand-in); the address is looked up once per device with
// cudaGetSymbolAddress, with that device current.
namespace {

constexpr int64_t kStaticStagingBytes = int64_t(32) << 20;
std::mutex g_static_mutex;
void *g_static_staging_addr[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_static_staging[kStaticStagingBytes];

extern "C" int rope_qk_host_static(const rope_qk_desc *desc, void *stream)
{
    int rc = check_host_call(desc);
    if (rc != ROPE_OK) return rc;
    const rope_qk_desc &p = *desc;
    const int64_t T = p.total_tokens;
    if (T == 0) return ROPE_OK;
    const int64_t q_row = static_cast<int64_t>(p.n_q_heads) * p.head_dim * 2;
    const int64_t k_row = static_cast<int64_t>(p.n_kv_heads) * p.head_dim * 2;
    // one chunk must hold at least one token's Q and K rows
    if (q_row + k_row > kStaticStagingBytes) return ROPE_ERR_WORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ROPE_ERR_LAUNCH;
    void *staging = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mutex);
        if (g_static_staging_addr[dev] == nullptr) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_static_staging) != cudaSuccess || addr == nullptr)
                return ROPE_ERR_LAUNCH;
            g_static_staging_addr[dev] = addr;
        }
        staging = g_static_staging_addr[dev];
    }

    // one slot, everything in order on the caller's stream: copy a chunk in, rotate it,
    // copy it out, next chunk
    int64_t chunk = kStaticStagingBytes / (q_row + k_row);
    if (chunk > T) chunk = T;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *const dq = static_cast<char *>(staging);
    char *const dk = dq + chunk * q_row;
    char *const q_host = static_cast<char *>(p.q);
    char *const k_host = static_cast<char *>(p.k);
    char *const qo_host = static_cast<char *>(p.q_out != nullptr ? p.q_out : p.q);
    char *const ko_host = static_cast<char *>(p.k_out != nullptr ? p.k_out : p.k);
    for (int64_t t0 = 0; t0 < T; t0 += chunk) {
        const int64_t n = (T - t0) < chunk ? (T - t0) : chunk;
        if (cudaMemcpyAsync(dq, q_host + t0 * q_row, n * q_row, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(dk, k_host + t0 * k_row, n * k_row, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return ROPE_ERR_LAUNCH;
        rope_qk_segment segs[ROPE_MAX_SEGMENTS];
        const rope_qk_desc cd = chunk_desc(p, t0, n, dq, dk, segs);
        rc = rope_qk_apply_plain_launch(&cd, stream);
        if (rc != ROPE_OK) return rc;
        if (cudaMemcpyAsync(qo_host + t0 * q_row, dq, n * q_row, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaMemcpyAsync(ko_host + t0 * k_row, dk, n * k_row, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return ROPE_ERR_LAUNCH;
    }
    return ROPE_OK;
}
