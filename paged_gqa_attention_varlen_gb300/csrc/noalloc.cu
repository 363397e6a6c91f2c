// noalloc.cu -- a paged decode entry point that allocates nothing.
//
// pgqa_paged_decode_bf16 keeps its split-KV partial results in a library workspace that
// it cudaMalloc's on first use.  Some callers cannot allow that: engines that hand every
// byte of free device memory to their own pool allocator at start-up (a later cudaMalloc
// fails or fragments the pool), and hosts that forbid allocation after initialisation
// (real-time or certified deployments).  This file gives them
// pgqa_paged_decode_bf16_noalloc, which runs the same plan / split-KV / merge kernels but
// keeps their scratch in one fixed-size array in the library's own device memory.
//
// The array is a file-scope static __device__ object of kNoAllocScratchBytes: every GPU
// that loads the library holds it until the process exits.  In host code its name is
// only a host-side stand-in, so the first call on each device resolves the device
// address with cudaGetSymbolAddress (with that device current) and passes it to the
// kernels.  The status word the
// kernels write lives in the array too, so device-side errors of this call (skipped bad
// page ids, an expired bounded wait) are not reported to the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pgqa.h"
#include "internal.h"

namespace pgqa {
namespace decode {
cudaError_t launch_plan(const PlanParams&, cudaStream_t);
cudaError_t launch_decode(const Params&, int group, int num_sms, cudaStream_t);
cudaError_t launch_merge(const Params&, cudaStream_t);
cudaError_t prepare_page_maps(Params&, const void*, const void*, int, int, int, long long,
                              long long, long long, bool);
}  // namespace decode

namespace {

// Maximum scratch of the allocation-free decode: 16 MiB.  It bounds
// batch * ceil(page_table_stride * page_size / 1024) * num_qo_heads * (head_dim + 1) floats
// of partial results plus two int arrays of about batch entries.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
constexpr size_t kScratchHeader = 1024;  // status word + padding

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
struct Slot {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    unsigned char* addr = nullptr;  // device address of g_noalloc_scratch on this device
};
std::mutex g_lock;
Slot g_slots[kMaxDev];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of scratch a call with these sizes needs (same carving as the kernels use below).
size_t scratch_needed(int batch, int stride, int page_size, int hq, int d, int hk,
                      long long* chunks, int* chunk) {
    const long long max_kv = (long long)stride * page_size;
    *chunk = decode::chunk_keys(batch, max_kv, hk);
    *chunks = decode::total_chunks(batch, max_kv, *chunk);
    return kScratchHeader + round256((size_t)(2 * batch + 1) * sizeof(int)) +
           round256((size_t)*chunks * hq * sizeof(float)) + (size_t)*chunks * hq * d * sizeof(float);
}

}  // namespace
}  // namespace pgqa

using namespace pgqa;

extern "C" int pgqa_paged_decode_bf16_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
    const int32_t* kv_lens, int page_size, int page_table_stride, int num_pages, void* o,
    float* lse, int batch, int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale,
    pgqa_stream_t stream) {
    if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || page_table_stride < 0 ||
        num_pages < 0)
        return PGQA_ERR_INVALID_ARG;
    if (batch == 0) return PGQA_OK;
    if (!q || !k_pages || !v_pages || !o || !kv_lens || (!page_table && page_table_stride > 0))
        return PGQA_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(q) || !a16(k_pages) || !a16(v_pages) || !a16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
        return PGQA_ERR_INVALID_ARG;
    if (head_dim != decode::HEAD_DIM) return PGQA_ERR_UNSUPPORTED;
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
        return PGQA_ERR_UNSUPPORTED;
    if (num_qo_heads % num_kv_heads != 0) return PGQA_ERR_UNSUPPORTED;
    const int group = num_qo_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PGQA_ERR_UNSUPPORTED;
    if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
        return PGQA_ERR_INVALID_ARG;
    if ((long long)page_table_stride * page_size > 0x7fffffffLL) return PGQA_ERR_UNSUPPORTED;

    // Sizes beyond the fixed scratch are rejected before anything is enqueued.
    long long chunks = 0;
    int chunk = decode::CHUNK;
    const size_t need = scratch_needed(batch, page_table_stride, page_size, num_qo_heads, head_dim,
                                       num_kv_heads, &chunks, &chunk);
    if (need > kNoAllocScratchBytes) return PGQA_ERR_WORKSPACE;

    std::lock_guard<std::mutex> guard(g_lock);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return PGQA_ERR_NO_DEVICE;
    }
    Slot& s = g_slots[dev];
    if (!s.ready) {
        // One-time set-up on this device (the device is current): architecture check and
        // the device address of the static scratch array.
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return PGQA_ERR_NO_DEVICE;
        }
        s.supported = prop.major == 10 && prop.minor == 3;
        s.num_sms = prop.multiProcessorCount;
        if (s.supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                return PGQA_ERR_CUDA;
            }
            s.addr = static_cast<unsigned char*>(addr);
        }
        s.ready = true;
    }
    if (!s.supported) return PGQA_ERR_NO_DEVICE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned char* base = s.addr;
    int* status = reinterpret_cast<int*>(base);
    // The array keeps the previous call's contents: the status word must start at zero;
    // every other byte a kernel reads is written earlier in the same call.
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return PGQA_ERR_CUDA;
    int* chunk_off = reinterpret_cast<int*>(base + kScratchHeader);
    int* kv_eff = chunk_off + (batch + 1);
    const size_t lse_off = kScratchHeader + round256((size_t)(2 * batch + 1) * sizeof(int));
    float* part_lse = reinterpret_cast<float*>(base + lse_off);
    float* part_o = reinterpret_cast<float*>(
        base + lse_off + round256((size_t)chunks * num_qo_heads * sizeof(float)));

    decode::PlanParams pp;
    pp.kv_lens = kv_lens;
    pp.kv_eff = kv_eff;
    pp.chunk_off = chunk_off;
    pp.status = status;
    pp.batch = batch;
    pp.max_kv = page_table_stride * page_size;
    pp.chunk = chunk;
    pp.q_indptr = nullptr;  // one query row per request
    pp.q_off = nullptr;
    pp.q_len = nullptr;
    pp.max_qo = 1;
    if (decode::launch_plan(pp, st) != cudaSuccess) return PGQA_ERR_CUDA;

    decode::Params p;
    p.q = q;
    p.k_pages = k_pages;
    p.v_pages = v_pages;
    p.page_table = page_table;
    p.kv_eff = kv_eff;
    p.chunk_off = chunk_off;
    p.o = o;
    p.lse = lse;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.status = status;
    p.batch = batch;
    p.page_table_stride = page_table_stride;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = num_kv_heads;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    p.q_off = nullptr;
    p.q_len = nullptr;
    p.max_qo = 1;
    p.causal = 1;
    p.chunk_capacity = chunks;
    p.chunk = chunk;
    if (decode::prepare_page_maps(p, k_pages, v_pages, num_pages, num_kv_heads, page_size,
                                  (long long)page_size * num_kv_heads * head_dim,
                                  (long long)num_kv_heads * head_dim, head_dim, false) != cudaSuccess)
        return PGQA_ERR_INVALID_ARG;
    if (decode::launch_decode(p, group, s.num_sms, st) != cudaSuccess) return PGQA_ERR_CUDA;
    return decode::launch_merge(p, st) == cudaSuccess ? PGQA_OK : PGQA_ERR_CUDA;
}
