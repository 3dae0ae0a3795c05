// Host-buffer streaming for packed QK-RoPE: Q and K live in (pinned) host memory; the
// library walks the pack in chunks of tokens through a device staging workspace,
// overlapping the host-to-device copy of chunk i+1, the rotation of chunk i and the
// device-to-host copy of chunk i-1 on three streams.  Each chunk is rotated by the
// same kernel as rope_qk_apply with its global token offset (or its slice of the
// position ids), so the results are those of one rotation of the whole pack.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "rope_qk.h"

// rope_qk_apply with plain (not programmatically overlapped) launches (rope_qk.cu).
int rope_qk_apply_plain_launch(const rope_qk_desc *desc, void *stream);

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

// The position ids of rows [t0, ...) of a chunk: int32 or, with the flag, int64 values.
const int32_t *ids_from(const rope_qk_desc &p, int64_t t0)
{
    if ((p.flags & ROPE_FLAG_POSITION_IDS_INT64) != 0)
        return reinterpret_cast<const int32_t *>(reinterpret_cast<const int64_t *>(p.position_ids) + t0);
    return p.position_ids + t0;
}

}  // namespace

// Shared by rope_qk_host and its static-workspace variant: stream the pack through
// `workspace` (device, workspace_bytes) on `stream`.
int rope_qk_host_impl(const rope_qk_desc *dp, void *workspace, int64_t workspace_bytes, void *stream)
{
    if (dp == nullptr) return ROPE_ERR_NULL;
    const rope_qk_desc &p = *dp;
    const int64_t T = p.total_tokens;
    if (T < 0 || p.n_q_heads < 1 || p.n_kv_heads < 1 || p.token_offset < 0 || workspace_bytes < 0)
        return ROPE_ERR_SHAPE;
    if ((p.flags & ~ROPE_FLAG_POSITION_IDS_INT64) != 0) return ROPE_ERR_UNSUPPORTED;
    if (p.head_dim < 16 || p.head_dim > 256 || p.head_dim % 16 != 0) return ROPE_ERR_HEAD_DIM;
    if (T == 0) return ROPE_OK;
    if (p.q == nullptr || p.k == nullptr || workspace == nullptr) return ROPE_ERR_NULL;
    if ((p.q_out == nullptr) != (p.k_out == nullptr)) return ROPE_ERR_NULL;
    const int32_t d = p.head_dim;
    if (!contiguous(p.q, p.q_stride_token, p.q_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k, p.k_stride_token, p.k_stride_head, p.n_kv_heads, d) ||
        !contiguous(p.q_out, p.q_out_stride_token, p.q_out_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k_out, p.k_out_stride_token, p.k_out_stride_head, p.n_kv_heads, d))
        return ROPE_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ROPE_ERR_ALIGN;
    // what rope_qk_apply would reject for the whole pack is rejected before any copy
    if (!(p.theta > 0.0) || p.theta > 1.7e308 || !(p.position_scale > 0.0) || p.position_scale > 1.7e308)
        return ROPE_ERR_THETA;
    if (p.position_ids == nullptr && p.cu_seqlens == nullptr) return ROPE_ERR_NULL;
    if (p.position_ids == nullptr && (p.n_seqs < 0 || p.token_offset + T > (int64_t(1) << 24)))
        return p.n_seqs < 0 ? ROPE_ERR_SHAPE : ROPE_ERR_UNSUPPORTED;
    if (p.cos_sin_cache != nullptr && (reinterpret_cast<uintptr_t>(p.cos_sin_cache) & 15u) != 0) return ROPE_ERR_ALIGN;
    if (p.cache_rows < 0) return ROPE_ERR_SHAPE;

    // chunk geometry: two slots, each holding the Q and K rows of `chunk` tokens
    const int64_t q_row = static_cast<int64_t>(p.n_q_heads) * d * 2;
    const int64_t k_row = static_cast<int64_t>(p.n_kv_heads) * d * 2;
    const int64_t per_token = q_row + k_row;
    int64_t chunk = workspace_bytes / (kSlots * per_token);
    chunk -= chunk % 8;                       // keep every slot's K part 16-byte aligned
    if (chunk < 8) return ROPE_ERR_UNSUPPORTED;
    if (chunk > T) chunk = T;
    const int64_t slot_bytes = ((chunk * per_token) + 255) / 256 * 256;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceQueues *qs = nullptr;
    int rc = queues_for_current_device(&qs);
    if (rc != ROPE_OK) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // On an early return the caller's stream still waits for every copy already queued,
    // so that freeing or reusing the workspace or the host buffers after the error is
    // ordered after them.
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
        rope_qk_desc cd = p;
        cd.q = dq;
        cd.k = dk;
        cd.q_stride_token = p.n_q_heads * static_cast<int64_t>(d);
        cd.q_stride_head = d;
        cd.k_stride_token = p.n_kv_heads * static_cast<int64_t>(d);
        cd.k_stride_head = d;
        cd.q_out = nullptr;
        cd.k_out = nullptr;
        cd.total_tokens = n;
        if (p.position_ids != nullptr) cd.position_ids = ids_from(p, t0);
        else cd.token_offset = p.token_offset + t0;
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
    if (desc == nullptr) return ROPE_ERR_NULL;
    const rope_qk_desc &p = *desc;
    if (p.total_tokens < 0 || p.n_q_heads < 1 || p.n_kv_heads < 1) return ROPE_ERR_SHAPE;
    if ((p.flags & ~ROPE_FLAG_POSITION_IDS_INT64) != 0) return ROPE_ERR_UNSUPPORTED;
    if (p.head_dim < 16 || p.head_dim > 256 || p.head_dim % 16 != 0) return ROPE_ERR_HEAD_DIM;
    if (p.total_tokens == 0) return ROPE_OK;
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
    if (p.q == nullptr || p.k == nullptr) return ROPE_ERR_NULL;
    if ((p.q_out == nullptr) != (p.k_out == nullptr)) return ROPE_ERR_NULL;
    const int32_t d = p.head_dim;
    if (!contiguous(p.q, p.q_stride_token, p.q_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k, p.k_stride_token, p.k_stride_head, p.n_kv_heads, d) ||
        !contiguous(p.q_out, p.q_out_stride_token, p.q_out_stride_head, p.n_q_heads, d) ||
        !contiguous(p.k_out, p.k_out_stride_token, p.k_out_stride_head, p.n_kv_heads, d))
        return ROPE_ERR_SHAPE;

    // one slot, everything in order on the caller's stream: copy a chunk in, rotate it,
    // copy it out, next chunk
    const int64_t T = p.total_tokens;
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
        rope_qk_desc cd = p;
        cd.q = dq;
        cd.k = dk;
        cd.q_stride_token = q_row / 2;
        cd.q_stride_head = d;
        cd.k_stride_token = k_row / 2;
        cd.k_stride_head = d;
        cd.q_out = nullptr;
        cd.k_out = nullptr;
        cd.total_tokens = n;
        if (p.position_ids != nullptr) cd.position_ids = ids_from(p, t0);
        else cd.token_offset = p.token_offset + t0;
        const int rc = rope_qk_apply_plain_launch(&cd, stream);
        if (rc != ROPE_OK) return rc;
        if (cudaMemcpyAsync(qo_host + t0 * q_row, dq, n * q_row, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaMemcpyAsync(ko_host + t0 * k_row, dk, n * k_row, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return ROPE_ERR_LAUNCH;
    }
    return ROPE_OK;
}
