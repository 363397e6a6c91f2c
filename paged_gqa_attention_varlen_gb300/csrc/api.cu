// api.cu -- the C ABI of libpgqa (declared in include/pgqa.h): argument checks,
// per-device workspace, TMA tensor-map templates, and the kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pgqa.h"
#include "internal.h"

namespace pgqa {
namespace prefill {
cudaError_t launch_plan(const PlanParams&, const CUtensorMap&, const CUtensorMap&,
                        const CUtensorMap&, cudaStream_t);
template <int D, bool PAGED>
cudaError_t launch_attention(const Params&, int, bool grouped, cudaStream_t);
template <bool PAGED>
cudaError_t launch_attention_pair(const Params&, int, cudaStream_t);
cudaError_t launch_merge(const Params&, int head_dim, int num_sms, cudaStream_t);
}  // namespace prefill
namespace decode {
cudaError_t launch_plan(const PlanParams&, cudaStream_t);
cudaError_t launch_decode(const Params&, int group, int num_sms, cudaStream_t);
cudaError_t launch_merge(const Params&, cudaStream_t);
cudaError_t launch_decode_mma(const Params&, int group, int num_sms, cudaStream_t);
cudaError_t prepare_page_maps(Params&, const void*, const void*, int, int, int, long long,
                              long long, long long, bool);
}  // namespace decode
namespace dequant {
cudaError_t launch_dequant(const Params&, int num_sms, cudaStream_t);
}  // namespace dequant
namespace selftest {
cudaError_t launch_expired_wait(int* status, cudaStream_t stream);
}  // namespace selftest

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    bool ws_owned = false;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int map_cuda(cudaError_t e) { return e == cudaSuccess ? PGQA_OK : PGQA_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device, its properties (cached) and whether it is an sm_103 part.
int current_device(int* dev_out, DeviceState** st_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return PGQA_ERR_NO_DEVICE;
    }
    DeviceState& st = g_dev[dev];
    if (!st.probed) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return PGQA_ERR_NO_DEVICE;
        }
        st.supported = prop.major == 10 && prop.minor == 3;
        st.num_sms = prop.multiProcessorCount;
        st.probed = true;
    }
    if (!st.supported) return PGQA_ERR_NO_DEVICE;
    *dev_out = dev;
    *st_out = &st;
    return PGQA_OK;
}

int get_encoder() {
    if (g_encode) return PGQA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return PGQA_ERR_CUDA;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return PGQA_OK;
}

// Make sure the device workspace holds at least `need` bytes.  Allocation happens only
// outside stream capture; a fresh buffer starts with a cleared header.
int ensure_workspace(DeviceState& st, size_t need, cudaStream_t stream) {
    if (st.ws != nullptr && st.ws_bytes >= need) return PGQA_OK;
    if (st.ws != nullptr && !st.ws_owned) return PGQA_ERR_WORKSPACE;  // caller buffer too small
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return PGQA_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return PGQA_ERR_WORKSPACE;
    size_t bytes = need > kDefaultWorkspace ? align_up(need, 1u << 20) : kDefaultWorkspace;
    // a status still pending from an earlier call (and its diagnostic words) moves to the
    // new buffer rather than being lost with the old one
    WsHeader keep{};
    bool carry = false;
    if (st.ws != nullptr) {
        // Every kernel that may still set a status bit in the old buffer must finish before
        // its header is read: a blocking copy orders itself only against the legacy default
        // stream, not against the caller's non-blocking streams.
        if (cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            return PGQA_ERR_CUDA;
        }
        carry = cudaMemcpy(&keep, st.ws, sizeof(WsHeader), cudaMemcpyDeviceToHost) == cudaSuccess &&
                keep.status != 0;
        cudaGetLastError();
        cudaFree(st.ws);
        st.ws = nullptr;
        st.ws_bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return PGQA_ERR_WORKSPACE;
    }
    if (cudaMemset(p, 0, kWsArrays) != cudaSuccess) {
        cudaFree(p);
        return PGQA_ERR_CUDA;
    }
    if (carry) {
        WsHeader h{};
        const int* from = reinterpret_cast<const int*>(&keep);
        int* to = reinterpret_cast<int*>(&h);
        to[0] = from[0];  // the status word
        for (int i = kDiagFlag; i < kDiagFlag + kDiagWords; ++i) to[i] = from[i];
        if (cudaMemcpy(p, &h, sizeof(WsHeader), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(p);
            return PGQA_ERR_CUDA;
        }
    }
    st.ws = p;
    st.ws_bytes = bytes;
    st.ws_owned = true;
    return PGQA_OK;
}

int encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGQA_OK : PGQA_ERR_INVALID_ARG;
}

int encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGQA_OK : PGQA_ERR_INVALID_ARG;
}

// 4-D {d, slot, head, page} view of a page pool (element strides, d contiguous), box of
// 64 columns x page_size slots of one head, 128-byte swizzle (the prefill's stage layout).
int encode_pages_4d(CUtensorMap* map, const void* base, int d, int page_size, int heads,
                    int num_pages, long long page_stride, long long slot_stride,
                    long long head_stride) {
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)page_size, (cuuint64_t)heads,
                                (cuuint64_t)(num_pages > 0 ? num_pages : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)slot_stride * 2, (cuuint64_t)head_stride * 2,
                                   (cuuint64_t)page_stride * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)page_size, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGQA_OK : PGQA_ERR_INVALID_ARG;
}

// 5-D views of a page pool for the grouped stage layout; a box lands as 8-row swizzle atoms
// of each 64-column chunk 1 KB apart (the chunk dimension's stride is 128 bytes: the
// head_dim row of a slot is contiguous), groups of 8 rows (d / 64) KB apart.
//  - box_keys 16, when a page's (page, head) pairs are one dimension (page_stride a
//    multiple of head_stride, page_heads = page_stride / head_stride >= heads):
//    {64 columns, 8 slots, chunk, page_size / 8 halves, page * page_heads + head}, box
//    {64, 8, d / 64, 2, 1} = 16 slots of one page and head;
//  - box_keys 8 otherwise: {64 columns, slot, chunk, head, page}, box {64, 8, d / 64, 1, 1}.
int encode_pages_grouped(CUtensorMap* map, const void* base, int d, int page_size, int heads,
                         int num_pages, long long page_stride, long long slot_stride,
                         long long head_stride, int* box_keys, int* page_heads) {
    const long long np = num_pages > 0 ? num_pages : 1;
    const long long ph = page_stride % head_stride == 0 ? page_stride / head_stride : 0;
    const bool merged = ph >= heads && np * ph < (1LL << 31);
    cuuint64_t dims[5];
    cuuint64_t strides[4];
    cuuint32_t box[5];
    if (merged) {
        const cuuint64_t dd[5] = {64, 8, (cuuint64_t)(d / 64), (cuuint64_t)(page_size / 8),
                                  (cuuint64_t)(np * ph)};
        const cuuint64_t ss[4] = {(cuuint64_t)slot_stride * 2, 128, (cuuint64_t)slot_stride * 16,
                                  (cuuint64_t)head_stride * 2};
        const cuuint32_t bb[5] = {64, 8, (cuuint32_t)(d / 64), 2, 1};
        for (int i = 0; i < 5; ++i) dims[i] = dd[i], box[i] = bb[i];
        for (int i = 0; i < 4; ++i) strides[i] = ss[i];
    } else {
        const cuuint64_t dd[5] = {64, (cuuint64_t)page_size, (cuuint64_t)(d / 64), (cuuint64_t)heads,
                                  (cuuint64_t)np};
        const cuuint64_t ss[4] = {(cuuint64_t)slot_stride * 2, 128, (cuuint64_t)head_stride * 2,
                                  (cuuint64_t)page_stride * 2};
        const cuuint32_t bb[5] = {64, 8, (cuuint32_t)(d / 64), 1, 1};
        for (int i = 0; i < 5; ++i) dims[i] = dd[i], box[i] = bb[i];
        for (int i = 0; i < 4; ++i) strides[i] = ss[i];
    }
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *box_keys = merged ? 16 : 8;
    *page_heads = merged ? (int)ph : 0;
    return r == CUDA_SUCCESS ? PGQA_OK : PGQA_ERR_INVALID_ARG;
}

// Element strides of a page pool: positive multiples of 16 bytes (the TMA rule for
// global strides) and below 2^36 elements; elem_bytes is 2 (bf16) or 1 (E4M3).
bool kv_strides_ok(long long page_stride, long long slot_stride, long long head_stride,
                   int elem_bytes = 2) {
    const long long lim = 1LL << 36;
    for (long long x : {page_stride, slot_stride, head_stride})
        if (x <= 0 || ((x * elem_bytes) & 15) || x >= lim) return false;
    return true;
}

// Prefill workspace: seven per-request int arrays, then the work list, then the split-KV
// partial results (lse [rows] and O [rows, d] fp32) in what remains.
constexpr int kPrefillArrays = 7;

size_t prefill_ws_bytes(int batch, long long max_items) {
    const size_t arr = align_up((size_t)(batch + 1) * sizeof(int), 256);
    return kWsArrays + kPrefillArrays * arr + (size_t)max_items * sizeof(prefill::WorkItem);
}

struct PrefillWs {
    WsHeader* hdr;
    CUtensorMap* tmaps;
    int *tile_off, *kv_off, *unit_off, *part_off, *merge_off, *nch, *kvl;
    prefill::WorkItem* items;
    long long item_capacity;
    float *part_lse, *part_o;
    long long part_capacity;
};

// Carve the first `usable` bytes of the workspace (all of it by default): a quarter of the
// space after the arrays holds the work list (at least what 4096 items need), the rest the
// partial results.
PrefillWs prefill_layout(const DeviceState& st, int batch, int head_dim, size_t usable = 0) {
    PrefillWs w;
    uint8_t* ws = static_cast<uint8_t*>(st.ws);
    const size_t ws_bytes = usable != 0 ? usable : st.ws_bytes;
    w.hdr = reinterpret_cast<WsHeader*>(ws + kWsHeader);
    w.tmaps = reinterpret_cast<CUtensorMap*>(ws + kWsTmapOffset);
    const size_t arr = align_up((size_t)(batch + 1) * sizeof(int), 256);
    int** arrays[kPrefillArrays] = {&w.tile_off, &w.kv_off, &w.unit_off, &w.part_off,
                                    &w.merge_off, &w.nch, &w.kvl};
    for (int i = 0; i < kPrefillArrays; ++i)
        *arrays[i] = reinterpret_cast<int*>(ws + kWsArrays + i * arr);
    const size_t items_off = kWsArrays + kPrefillArrays * arr;
    const size_t rest = ws_bytes > items_off ? ws_bytes - items_off : 0;
    size_t item_bytes = align_up(rest / 4, 256);
    const size_t min_items = 4096 * sizeof(prefill::WorkItem);
    if (item_bytes < min_items) item_bytes = rest < min_items ? rest : min_items;
    w.items = reinterpret_cast<prefill::WorkItem*>(ws + items_off);
    w.item_capacity = (long long)(item_bytes / sizeof(prefill::WorkItem));
    const size_t part_off = items_off + item_bytes;
    const size_t part_bytes = ws_bytes > part_off + 256 ? ws_bytes - part_off - 256 : 0;
    const long long rows = (long long)(part_bytes / ((size_t)(head_dim + 1) * sizeof(float)));
    w.part_capacity = rows;
    w.part_lse = reinterpret_cast<float*>(ws + part_off);
    w.part_o = reinterpret_cast<float*>(ws + part_off + align_up((size_t)rows * sizeof(float), 256));
    if (rows > 0 && align_up((size_t)rows * sizeof(float), 256) + (size_t)rows * head_dim * 4 >
                        part_bytes + 256)
        w.part_capacity = rows - 64;  // keep the O block inside the workspace
    if (w.part_capacity < 0) w.part_capacity = 0;
    return w;
}

// Plan and attention parameters shared by the ragged and paged prefill
void fill_split(prefill::PlanParams& pp, prefill::Params& p, const PrefillWs& w, int batch,
                int head_dim, int num_qo_heads, int num_sms) {
    pp.split_ok = 1;
    pp.split_tiles = p.split_tiles = head_dim == 256 ? 32 : 16;
    pp.num_ctas = num_sms;
    pp.num_qo_heads = num_qo_heads;
    pp.part_capacity = w.part_capacity;
    pp.unit_off = w.unit_off;
    pp.part_off = w.part_off;
    pp.merge_off = w.merge_off;
    pp.nch = w.nch;
    pp.kvl = w.kvl;
    p.part_o = w.part_o;
    p.part_lse = w.part_lse;
    p.merge_off = w.merge_off;
    p.part_off = w.part_off;
    p.nch = w.nch;
    p.kvl = w.kvl;
    p.batch = batch;
}

// Decode workspace: chunk offsets and kv lengths (plus query offsets and lengths when the
// requests have several query rows), then the partial lse and outputs of every chunk with
// room for max_qo query rows each.
size_t decode_ints(int batch, bool rows) { return (size_t)((rows ? 4 : 2) * (size_t)batch + 1); }
size_t decode_ws_bytes(int batch, int stride, int page_size, int hq, int d, int hk, bool rows,
                       int max_qo, int chunk_top = decode::CHUNK) {
    const long long max_kv = (long long)stride * page_size;
    const long long chunks =
        decode::total_chunks(batch, max_kv, decode::chunk_keys(batch, max_kv, hk, chunk_top));
    const size_t slots = (size_t)chunks * max_qo * hq;
    const size_t ints = align_up(decode_ints(batch, rows) * sizeof(int), 256);
    return kWsArrays + ints + align_up(slots * sizeof(float), 256) + slots * d * sizeof(float);
}

}  // namespace
}  // namespace pgqa

using namespace pgqa;

namespace {
int paged_decode_impl(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* page_table, const int32_t* kv_lens, int page_size,
                      int page_table_stride, int num_pages, int64_t page_stride,
                      int64_t slot_stride, int64_t head_stride, void* o, float* lse, int batch,
                      int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale, bool kv8,
                      float k_scale, float v_scale, const int32_t* q_indptr, int max_qo,
                      int causal, pgqa_stream_t stream);
int paged_prefill_impl(const void* q, const void* k_pages, const void* v_pages, void* o,
                       float* lse, const int32_t* q_indptr, const int32_t* page_table,
                       int page_table_stride, const int32_t* kv_lens, int page_size,
                       int num_pages, int64_t page_stride, int64_t slot_stride,
                       int64_t head_stride, int batch, int num_qo_heads, int num_kv_heads,
                       int head_dim, int causal, float sm_scale, bool kv8, float k_scale,
                       float v_scale, pgqa_stream_t stream);
}  // namespace

extern "C" {

int pgqa_version(void) { return 10000; }

const char* pgqa_status_string(int s) {
    switch (s) {
        case PGQA_OK: return "ok";
        case PGQA_ERR_INVALID_ARG: return "invalid argument";
        case PGQA_ERR_UNSUPPORTED: return "unsupported shape";
        case PGQA_ERR_WORKSPACE: return "workspace too small (allocation not allowed)";
        case PGQA_ERR_CUDA: return "CUDA error";
        case PGQA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case PGQA_ERR_DEVICE_BOUNDS: return "bad index data seen on the device";
        case PGQA_ERR_NO_DEVICE: return "no usable sm_103 device";
        case PGQA_ERR_DEVICE_CAPACITY: return "work list larger than the workspace";
        default: return "unknown status";
    }
}

size_t pgqa_workspace_bytes_prefill(int batch, int64_t max_total_q, int num_qo_heads,
                                    int num_kv_heads) {
    if (batch < 0 || max_total_q < 0 || num_kv_heads <= 0 || num_qo_heads <= 0) return 0;
    const long long g = num_qo_heads / num_kv_heads;
    const long long tiles = (max_total_q * g + prefill::BM - 1) / prefill::BM + batch;
    return prefill_ws_bytes(batch, tiles * num_kv_heads);
}

size_t pgqa_workspace_bytes_decode(int batch, int page_table_stride, int page_size,
                                   int num_qo_heads, int head_dim) {
    if (batch < 0 || page_table_stride < 0 || page_size <= 0 || num_qo_heads <= 0 ||
        head_dim <= 0)
        return 0;
    // an upper bound for any number of kv heads (one kv head gives the most chunks)
    return decode_ws_bytes(batch, page_table_stride, page_size, num_qo_heads, head_dim, 1, false,
                           1);
}

int pgqa_set_workspace(void* ptr, size_t bytes) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return PGQA_ERR_NO_DEVICE;
    }
    DeviceState& st = g_dev[dev];
    if (ptr != nullptr && ((reinterpret_cast<uintptr_t>(ptr) & 255u) != 0 || bytes < kWsArrays + 4096))
        return PGQA_ERR_INVALID_ARG;
    if (st.ws != nullptr && st.ws_owned) cudaFree(st.ws);
    st.ws = nullptr;
    st.ws_bytes = 0;
    st.ws_owned = false;
    if (ptr != nullptr) {
        if (cudaMemset(ptr, 0, kWsArrays) != cudaSuccess) {
            cudaGetLastError();
            return PGQA_ERR_CUDA;
        }
        st.ws = ptr;
        st.ws_bytes = bytes;
    }
    return PGQA_OK;
}

int pgqa_selftest_expired_wait(pgqa_stream_t stream) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev;
    DeviceState* st;
    int rc = current_device(&dev, &st);
    if (rc != PGQA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = ensure_workspace(*st, kWsArrays + 4096, s)) != PGQA_OK) return rc;
    return map_cuda(selftest::launch_expired_wait(static_cast<int*>(st->ws), s));
}

int pgqa_get_device_status(pgqa_stream_t stream) {
    std::lock_guard<std::mutex> lock(g_mutex);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PGQA_ERR_CUDA;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PGQA_ERR_NO_DEVICE;
    DeviceState& st = g_dev[dev];
    if (st.ws == nullptr) return PGQA_OK;
    int word = 0;
    if (cudaMemcpy(&word, st.ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return PGQA_ERR_CUDA;
    }
    if (word != 0) {  // clear the status word and the timeout diagnostic words
        const int zero = 0;
        cudaMemcpy(st.ws, &zero, sizeof(int), cudaMemcpyHostToDevice);
        cudaMemset(static_cast<int*>(st.ws) + kDiagFlag, 0, kDiagWords * sizeof(int));
    }
    if (word & PGQA_DEV_TIMEOUT) return PGQA_ERR_DEVICE_TIMEOUT;
    if (word & PGQA_DEV_BOUNDS) return PGQA_ERR_DEVICE_BOUNDS;
    if (word & PGQA_DEV_CAPACITY) return PGQA_ERR_DEVICE_CAPACITY;
    return PGQA_OK;
}

int pgqa_ragged_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* q_indptr, const int32_t* kv_indptr, int batch,
                             int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                             float sm_scale, pgqa_stream_t stream) {
    if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0) return PGQA_ERR_INVALID_ARG;
    if (batch == 0) return PGQA_OK;
    if (!q || !k || !v || !o || !q_indptr || !kv_indptr) return PGQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(q_indptr) & 3u) ||
        (reinterpret_cast<uintptr_t>(kv_indptr) & 3u))
        return PGQA_ERR_INVALID_ARG;
    if (head_dim != 128 && head_dim != 256) return PGQA_ERR_UNSUPPORTED;
    if (num_qo_heads % num_kv_heads != 0) return PGQA_ERR_UNSUPPORTED;
    const int group = num_qo_heads / num_kv_heads;
    if (group > prefill::BM || prefill::BM % group != 0) return PGQA_ERR_UNSUPPORTED;
    if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
        return PGQA_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    int dev;
    DeviceState* st;
    int rc = current_device(&dev, &st);
    if (rc != PGQA_OK) return rc;
    if ((rc = get_encoder()) != PGQA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // at least room for the tile offsets and a work list; the plan kernel checks the
    // list against what is there and reports overflow through the status word
    rc = ensure_workspace(*st, prefill_ws_bytes(batch, 4096), s);
    if (rc != PGQA_OK) return rc;

    const PrefillWs lay = prefill_layout(*st, batch, head_dim);
    WsHeader* hdr = lay.hdr;
    CUtensorMap* tmaps = lay.tmaps;
    int* tile_off = lay.tile_off;
    prefill::WorkItem* items = lay.items;
    const long long capacity = lay.item_capacity;

    // Tensor-map templates: row extents are placeholders (one box), patched on the
    // device from q_indptr[batch] / kv_indptr[batch] by the plan kernel.
    CUtensorMap tq, tk, tv;
    const uint32_t tpt = prefill::BM / group;
    if ((rc = encode_3d(&tq, q, head_dim, num_qo_heads, tpt, (uint64_t)head_dim * 2,
                        (uint64_t)num_qo_heads * head_dim * 2, 64, group, tpt)) != PGQA_OK)
        return rc;
    if ((rc = encode_2d(&tk, k, (uint64_t)num_kv_heads * head_dim, prefill::BN,
                        (uint64_t)num_kv_heads * head_dim * 2, 64, prefill::BN)) != PGQA_OK)
        return rc;
    if ((rc = encode_2d(&tv, v, (uint64_t)num_kv_heads * head_dim, prefill::BN,
                        (uint64_t)num_kv_heads * head_dim * 2, 64, prefill::BN)) != PGQA_OK)
        return rc;

    prefill::PlanParams pp;
    pp.q_indptr = q_indptr;
    pp.kv_indptr = kv_indptr;
    pp.kv_lens = nullptr;
    pp.max_kv = 0;
    pp.kv_off = nullptr;
    pp.batch = batch;
    pp.num_kv_heads = num_kv_heads;
    pp.group = group;
    pp.causal = causal ? 1 : 0;
    // hd128 runs two q tiles per work item (two softmax warpgroups share one K/V
    // stream); hd256 needs all of tensor memory for one tile
    pp.tiles_per_item = head_dim == 128 ? 2 : 1;
    pp.hdr = hdr;
    pp.tile_off = tile_off;
    pp.items = items;
    pp.item_capacity = capacity;
    pp.tm_out = tmaps;
    cudaError_t e;

    prefill::Params p;
    p.tm_q = tmaps + 0;
    p.tm_k = tmaps + 1;
    p.tm_v = tmaps + 2;
    p.o = o;
    p.lse = lse;
    p.q_indptr = q_indptr;
    p.kv_indptr = kv_indptr;
    p.items = items;
    p.hdr = hdr;
    p.status = &hdr->status;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    p.f8conv = 0;
    p.page_table = nullptr;
    p.page_table_stride = 0;
    p.page_size = 0;
    p.num_pages = 0;
    p.box_keys = 0;
    p.page_heads = 0;
    fill_split(pp, p, lay, batch, head_dim, num_qo_heads, st->num_sms);
    e = prefill::launch_plan(pp, tq, tk, tv, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;
    e = head_dim == 128 ? prefill::launch_attention_pair<false>(p, st->num_sms, s)
                        : prefill::launch_attention<256, false>(p, st->num_sms, false, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;
    return map_cuda(prefill::launch_merge(p, head_dim, st->num_sms, s));
}

int pgqa_paged_prefill_bf16(const void* q, const void* k_pages, const void* v_pages, void* o,
                            float* lse, const int32_t* q_indptr, const int32_t* page_table,
                            int page_table_stride, const int32_t* kv_lens, int page_size,
                            int num_pages, int batch, int num_qo_heads, int num_kv_heads,
                            int head_dim, int causal, float sm_scale, pgqa_stream_t stream) {
    const long long hd = (long long)num_kv_heads * head_dim;
    return pgqa_paged_prefill_bf16_strided(q, k_pages, v_pages, o, lse, q_indptr, page_table,
                                           page_table_stride, kv_lens, page_size, num_pages,
                                           hd * page_size, hd, head_dim, batch, num_qo_heads,
                                           num_kv_heads, head_dim, causal, sm_scale, stream);
}

int pgqa_paged_prefill_bf16_strided(const void* q, const void* k_pages, const void* v_pages,
                                    void* o, float* lse, const int32_t* q_indptr,
                                    const int32_t* page_table, int page_table_stride,
                                    const int32_t* kv_lens, int page_size, int num_pages,
                                    int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                                    int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                    int causal, float sm_scale, pgqa_stream_t stream) {
    return paged_prefill_impl(q, k_pages, v_pages, o, lse, q_indptr, page_table,
                              page_table_stride, kv_lens, page_size, num_pages, page_stride,
                              slot_stride, head_stride, batch, num_qo_heads, num_kv_heads,
                              head_dim, causal, sm_scale, false, 1.f, 1.f, stream);
}

int pgqa_paged_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* kv_lens, int page_size,
                           int page_table_stride, int num_pages, void* o, float* lse,
                           int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           float sm_scale, pgqa_stream_t stream) {
    const long long hd = (long long)num_kv_heads * head_dim;
    return pgqa_paged_decode_bf16_strided(q, k_pages, v_pages, page_table, kv_lens, page_size,
                                          page_table_stride, num_pages, hd * page_size, hd,
                                          head_dim, o, lse, batch, num_qo_heads, num_kv_heads,
                                          head_dim, sm_scale, stream);
}

int pgqa_paged_decode_bf16_strided(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, const int32_t* kv_lens,
                                   int page_size, int page_table_stride, int num_pages,
                                   int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                                   void* o, float* lse, int batch, int num_qo_heads,
                                   int num_kv_heads, int head_dim, float sm_scale,
                                   pgqa_stream_t stream) {
    return paged_decode_impl(q, k_pages, v_pages, page_table, kv_lens, page_size,
                             page_table_stride, num_pages, page_stride, slot_stride, head_stride,
                             o, lse, batch, num_qo_heads, num_kv_heads, head_dim, sm_scale, false,
                             1.f, 1.f, nullptr, 1, 1, stream);
}

static bool finite_scale(float x) { return x == x && x <= 3.0e38f && x >= -3.0e38f; }

int pgqa_paged_decode_e4m3(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* kv_lens, int page_size,
                           int page_table_stride, int num_pages, int64_t page_stride,
                           int64_t slot_stride, int64_t head_stride, float k_scale, float v_scale,
                           void* o, float* lse, int batch, int num_qo_heads, int num_kv_heads,
                           int head_dim, float sm_scale, pgqa_stream_t stream) {
    if (!finite_scale(k_scale) || !finite_scale(v_scale)) return PGQA_ERR_INVALID_ARG;
    return paged_decode_impl(q, k_pages, v_pages, page_table, kv_lens, page_size,
                             page_table_stride, num_pages, page_stride, slot_stride, head_stride,
                             o, lse, batch, num_qo_heads, num_kv_heads, head_dim, sm_scale, true,
                             k_scale, v_scale, nullptr, 1, 1, stream);
}

int pgqa_paged_prefill_e4m3(const void* q, const void* k_pages, const void* v_pages, void* o,
                            float* lse, const int32_t* q_indptr, const int32_t* page_table,
                            int page_table_stride, const int32_t* kv_lens, int page_size,
                            int num_pages, int64_t page_stride, int64_t slot_stride,
                            int64_t head_stride, float k_scale, float v_scale, int batch,
                            int max_qo_len, int num_qo_heads, int num_kv_heads, int head_dim,
                            int causal, float sm_scale, pgqa_stream_t stream) {
    if (!finite_scale(k_scale) || !finite_scale(v_scale)) return PGQA_ERR_INVALID_ARG;
    if (batch > 0 && (max_qo_len < 1 || !q_indptr)) return PGQA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q_indptr) & 3u) return PGQA_ERR_INVALID_ARG;
    // few query rows per request: the tensor-core E4M3 decode, with every request's rows as
    // the columns of its MMAs (the keys stream once for all of them)
    const int group = num_kv_heads > 0 && num_qo_heads % num_kv_heads == 0
                          ? num_qo_heads / num_kv_heads : 0;
    const bool few_rows = head_dim == 128 && (group == 1 || group == 2 || group == 4 ||
                                              group == 8) &&
                          (long long)max_qo_len * group <= 16;
    if (few_rows || batch == 0)
        return paged_decode_impl(q, k_pages, v_pages, page_table, kv_lens, page_size,
                                 page_table_stride, num_pages, page_stride, slot_stride,
                                 head_stride, o, lse, batch, num_qo_heads, num_kv_heads, head_dim,
                                 sm_scale, true, k_scale, v_scale, q_indptr, max_qo_len,
                                 causal ? 1 : 0, stream);
    // longer query runs: the bf16 prefill over the converted pages
    return paged_prefill_impl(q, k_pages, v_pages, o, lse, q_indptr, page_table,
                              page_table_stride, kv_lens, page_size, num_pages, page_stride,
                              slot_stride, head_stride, batch, num_qo_heads, num_kv_heads,
                              head_dim, causal, sm_scale, true, k_scale, v_scale, stream);
}

}  // extern "C"

namespace {
// The paged decode for bf16 (kv8 = false) or E4M3 (kv8 = true, with per-tensor scales)
// K/V pools of the given element strides.
int paged_decode_impl(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* page_table, const int32_t* kv_lens, int page_size,
                      int page_table_stride, int num_pages, int64_t page_stride,
                      int64_t slot_stride, int64_t head_stride, void* o, float* lse, int batch,
                      int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale, bool kv8,
                      float k_scale, float v_scale, const int32_t* q_indptr, int max_qo,
                      int causal, pgqa_stream_t stream) {
    if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || page_table_stride < 0 ||
        num_pages < 0)
        return PGQA_ERR_INVALID_ARG;
    if (batch > 0 && !kv_strides_ok(page_stride, slot_stride, head_stride, kv8 ? 1 : 2))
        return PGQA_ERR_INVALID_ARG;
    if (batch == 0) return PGQA_OK;
    if (!q || !k_pages || !v_pages || !o || !kv_lens || (!page_table && page_table_stride > 0))
        return PGQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
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

    std::lock_guard<std::mutex> lock(g_mutex);
    int dev;
    DeviceState* st;
    int rc = current_device(&dev, &st);
    if (rc != PGQA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool rows = q_indptr != nullptr;
    // the E4M3 tensor-core form with several query rows per request takes chunks of at
    // most 896 keys
    const int chunk_top = kv8 && max_qo > 1 ? decode::CHUNK_E4M3_ROWS : decode::CHUNK;
    const size_t need = decode_ws_bytes(batch, page_table_stride, page_size, num_qo_heads, head_dim,
                                        num_kv_heads, rows, max_qo, chunk_top);
    rc = ensure_workspace(*st, need, s);
    if (rc != PGQA_OK) return rc;

    uint8_t* ws = static_cast<uint8_t*>(st->ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + kWsHeader);
    int* chunk_off = reinterpret_cast<int*>(ws + kWsArrays);
    int* kv_eff = chunk_off + (batch + 1);
    int* q_off = rows ? kv_eff + batch : nullptr;
    int* q_len = rows ? q_off + batch : nullptr;
    const size_t lse_off = kWsArrays + align_up(decode_ints(batch, rows) * sizeof(int), 256);
    const long long max_kv = (long long)page_table_stride * page_size;
    const int chunk = decode::chunk_keys(batch, max_kv, num_kv_heads, chunk_top);
    const long long chunks = decode::total_chunks(batch, max_kv, chunk);
    float* part_lse = reinterpret_cast<float*>(ws + lse_off);
    float* part_o = reinterpret_cast<float*>(
        ws + lse_off + align_up((size_t)chunks * max_qo * num_qo_heads * sizeof(float), 256));

    decode::PlanParams pp;
    pp.kv_lens = kv_lens;
    pp.kv_eff = kv_eff;
    pp.chunk_off = chunk_off;
    pp.status = &hdr->status;
    pp.batch = batch;
    pp.max_kv = (int)max_kv;
    pp.chunk = chunk;
    pp.q_indptr = q_indptr;
    pp.q_off = q_off;
    pp.q_len = q_len;
    pp.max_qo = max_qo;
    cudaError_t e = decode::launch_plan(pp, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;

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
    p.status = &hdr->status;
    p.batch = batch;
    p.page_table_stride = page_table_stride;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = num_kv_heads;
    p.scale_log2 = sm_scale * 1.4426950408889634f * k_scale;
    p.v_scale = v_scale;
    p.q_off = q_off;
    p.q_len = q_len;
    p.max_qo = max_qo;
    p.causal = causal;
    p.chunk_capacity = chunks;
    p.chunk = chunk;
    if (decode::prepare_page_maps(p, k_pages, v_pages, num_pages, num_kv_heads, page_size,
                                  page_stride, slot_stride, head_stride, kv8) != cudaSuccess)
        return PGQA_ERR_INVALID_ARG;
    // E4M3 K/V: the dot products on the tensor cores (the CUDA cores convert bytes)
    e = kv8 ? decode::launch_decode_mma(p, group, st->num_sms, s)
            : decode::launch_decode(p, group, st->num_sms, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;
    return map_cuda(decode::launch_merge(p, s));
}

// The paged prefill over bf16 K/V pools (kv8 = false), or over E4M3 pools (kv8 = true):
// the pages the call reads are then converted into a bf16 pool at the end of the
// workspace first (dequant.cu), k_scale joins the score scale and v_scale the output
// scale.
int paged_prefill_impl(const void* q, const void* k_pages, const void* v_pages, void* o,
                       float* lse, const int32_t* q_indptr, const int32_t* page_table,
                       int page_table_stride, const int32_t* kv_lens, int page_size,
                       int num_pages, int64_t page_stride, int64_t slot_stride,
                       int64_t head_stride, int batch, int num_qo_heads, int num_kv_heads,
                       int head_dim, int causal, float sm_scale, bool kv8, float k_scale,
                       float v_scale, pgqa_stream_t stream) {
    if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || page_table_stride < 0 ||
        num_pages < 0)
        return PGQA_ERR_INVALID_ARG;
    if (batch > 0 && !kv_strides_ok(page_stride, slot_stride, head_stride, kv8 ? 1 : 2))
        return PGQA_ERR_INVALID_ARG;
    if (batch == 0) return PGQA_OK;
    if (!q || !k_pages || !v_pages || !o || !q_indptr || !kv_lens ||
        (!page_table && page_table_stride > 0))
        return PGQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(q_indptr) & 3u) ||
        (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
        return PGQA_ERR_INVALID_ARG;
    if (head_dim != 128 && head_dim != 256) return PGQA_ERR_UNSUPPORTED;
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
        return PGQA_ERR_UNSUPPORTED;
    if (num_qo_heads % num_kv_heads != 0) return PGQA_ERR_UNSUPPORTED;
    const int group = num_qo_heads / num_kv_heads;
    if (group > prefill::BM || prefill::BM % group != 0) return PGQA_ERR_UNSUPPORTED;
    if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
        return PGQA_ERR_INVALID_ARG;
    if ((long long)page_table_stride * page_size > 0x7fffffffLL) return PGQA_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_mutex);
    int dev;
    DeviceState* st;
    int rc = current_device(&dev, &st);
    if (rc != PGQA_OK) return rc;
    if ((rc = get_encoder()) != PGQA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // E4M3 pools: a bf16 pool of the pages the call reads (by page when the caller's pool is
    // the smaller, else by table slot with a rewritten table), after the prefill's own part
    const long long slots = (long long)batch * page_table_stride;
    const bool by_page = (long long)num_pages <= slots;
    long long pool_pages = by_page ? num_pages : slots;
    if (pool_pages < 1) pool_pages = 1;
    if (kv8 && pool_pages > 0x7fffffffLL) return PGQA_ERR_UNSUPPORTED;
    const size_t page_bytes = (size_t)page_size * num_kv_heads * head_dim * 2;
    const size_t pool_bytes = kv8 ? align_up((size_t)pool_pages * page_bytes, 1024) : 0;
    const size_t table_bytes = kv8 && !by_page ? align_up((size_t)slots * sizeof(int), 1024) : 0;
    const size_t tail = 2 * pool_bytes + table_bytes;
    size_t head_need = prefill_ws_bytes(batch, 4096);
    if (kv8 && head_need < kDefaultWorkspace) head_need = kDefaultWorkspace;
    head_need = align_up(head_need, 1024);
    rc = ensure_workspace(*st, head_need + tail, s);
    if (rc != PGQA_OK) return rc;

    const size_t usable = kv8 ? ((st->ws_bytes - tail) & ~(size_t)1023) : 0;
    const PrefillWs lay = prefill_layout(*st, batch, head_dim, usable);
    dequant::Params dq;  // E4M3 pools: launched right after the plan, beside it
    if (kv8) {
        uint8_t* tail_base = static_cast<uint8_t*>(st->ws) + usable;
        dq.k8 = static_cast<const uint8_t*>(k_pages);
        dq.v8 = static_cast<const uint8_t*>(v_pages);
        dq.page_stride = page_stride;
        dq.slot_stride = slot_stride;
        dq.head_stride = head_stride;
        dq.k16 = tail_base;
        dq.v16 = tail_base + pool_bytes;
        dq.page_table = page_table;
        dq.kv_lens = kv_lens;
        dq.table_out = by_page ? nullptr : reinterpret_cast<int*>(tail_base + 2 * pool_bytes);
        dq.status = &lay.hdr->status;
        dq.batch = batch;
        dq.page_table_stride = page_table_stride;
        dq.page_size = page_size;
        dq.num_pages = num_pages;
        dq.num_kv_heads = num_kv_heads;
        dq.head_dim = head_dim;
        // from here on the call reads the converted pool: packed NHD, pool_pages pages
        k_pages = dq.k16;
        v_pages = dq.v16;
        if (!by_page) page_table = dq.table_out;
        num_pages = (int)pool_pages;
        page_stride = (int64_t)page_size * num_kv_heads * head_dim;
        slot_stride = (int64_t)num_kv_heads * head_dim;
        head_stride = head_dim;
        sm_scale *= k_scale;
    }
    WsHeader* hdr = lay.hdr;
    CUtensorMap* tmaps = lay.tmaps;
    int* tile_off = lay.tile_off;
    int* kv_off = lay.kv_off;
    prefill::WorkItem* items = lay.items;
    const long long capacity = lay.item_capacity;

    // Q as for the ragged call (row extent patched on the device); K/V as 4-D page pools
    // {d, slot, head, page}, one box = one page of one head and one 64-column chunk.
    CUtensorMap tq, tk, tv;
    const uint32_t tpt = prefill::BM / group;
    if ((rc = encode_3d(&tq, q, head_dim, num_qo_heads, tpt, (uint64_t)head_dim * 2,
                        (uint64_t)num_qo_heads * head_dim * 2, 64, group, tpt)) != PGQA_OK)
        return rc;
    // head_dim 256 with pages of up to 32 tokens: the grouped stage layout (a 64 KB K/V tile
    // in 16 boxes of 4 KB rather than 4 * 128 / page_size boxes)
    const bool grouped = head_dim == 256 && page_size <= 32;
    int box_keys = 0, page_heads = 0;
    if (grouped) {
        if ((rc = encode_pages_grouped(&tk, k_pages, head_dim, page_size, num_kv_heads, num_pages,
                                       page_stride, slot_stride, head_stride, &box_keys,
                                       &page_heads)) != PGQA_OK ||
            (rc = encode_pages_grouped(&tv, v_pages, head_dim, page_size, num_kv_heads, num_pages,
                                       page_stride, slot_stride, head_stride, &box_keys,
                                       &page_heads)) != PGQA_OK)
            return rc;
    } else {
        if ((rc = encode_pages_4d(&tk, k_pages, head_dim, page_size, num_kv_heads, num_pages,
                                  page_stride, slot_stride, head_stride)) != PGQA_OK ||
            (rc = encode_pages_4d(&tv, v_pages, head_dim, page_size, num_kv_heads, num_pages,
                                  page_stride, slot_stride, head_stride)) != PGQA_OK)
            return rc;
    }

    prefill::PlanParams pp;
    pp.q_indptr = q_indptr;
    pp.kv_indptr = nullptr;
    pp.kv_lens = kv_lens;
    pp.max_kv = page_table_stride * page_size;
    pp.kv_off = kv_off;
    pp.batch = batch;
    pp.num_kv_heads = num_kv_heads;
    pp.group = group;
    pp.causal = causal ? 1 : 0;
    pp.tiles_per_item = head_dim == 128 ? 2 : 1;
    pp.hdr = hdr;
    pp.tile_off = tile_off;
    pp.items = items;
    pp.item_capacity = capacity;
    pp.tm_out = tmaps;
    cudaError_t e;

    prefill::Params p;
    p.tm_q = tmaps + 0;
    p.tm_k = tmaps + 1;
    p.tm_v = tmaps + 2;
    p.o = o;
    p.lse = lse;
    p.q_indptr = q_indptr;
    p.kv_indptr = nullptr;
    p.items = items;
    p.hdr = hdr;
    p.status = &hdr->status;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.v_scale = v_scale;
    p.f8conv = kv8 ? 1 : 0;  // pages converted from E4M3: V is f16
    p.page_table = page_table;
    p.page_table_stride = page_table_stride;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.box_keys = box_keys;
    p.page_heads = page_heads;
    fill_split(pp, p, lay, batch, head_dim, num_qo_heads, st->num_sms);
    e = prefill::launch_plan(pp, tq, tk, tv, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;
    // the plan needs nothing of the conversion (it reads q_indptr and kv_lens), and the
    // conversion nothing of the plan
    if (kv8 && dequant::launch_dequant(dq, st->num_sms, s) != cudaSuccess) return PGQA_ERR_CUDA;
    e = head_dim == 128 ? prefill::launch_attention_pair<true>(p, st->num_sms, s)
                        : prefill::launch_attention<256, true>(p, st->num_sms, grouped, s);
    if (e != cudaSuccess) return PGQA_ERR_CUDA;
    return map_cuda(prefill::launch_merge(p, head_dim, st->num_sms, s));
}
}  // namespace

extern "C" {

int ragged_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* q_indptr, const int32_t* kv_indptr, int batch,
                        int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                        float sm_scale, pgqa_stream_t stream) {
    return pgqa_ragged_prefill_bf16(q, k, v, o, lse, q_indptr, kv_indptr, batch, num_qo_heads,
                                    num_kv_heads, head_dim, causal, sm_scale, stream);
}

int paged_prefill_bf16(const void* q, const void* k_pages, const void* v_pages, void* o,
                       float* lse, const int32_t* q_indptr, const int32_t* page_table,
                       int page_table_stride, const int32_t* kv_lens, int page_size,
                       int num_pages, int batch, int num_qo_heads, int num_kv_heads,
                       int head_dim, int causal, float sm_scale, pgqa_stream_t stream) {
    return pgqa_paged_prefill_bf16(q, k_pages, v_pages, o, lse, q_indptr, page_table,
                                   page_table_stride, kv_lens, page_size, num_pages, batch,
                                   num_qo_heads, num_kv_heads, head_dim, causal, sm_scale, stream);
}

int paged_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* page_table, const int32_t* kv_lens, int page_size,
                      int page_table_stride, int num_pages, void* o, float* lse, int batch,
                      int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale,
                      pgqa_stream_t stream) {
    return pgqa_paged_decode_bf16(q, k_pages, v_pages, page_table, kv_lens, page_size,
                                  page_table_stride, num_pages, o, lse, batch, num_qo_heads,
                                  num_kv_heads, head_dim, sm_scale, stream);
}

}  // extern "C"
