// internal.h -- definitions shared by the host side and the kernels of libpgqa.
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

namespace pgqa {

// Device status word bits (first int of the workspace).
constexpr int PGQA_DEV_TIMEOUT = 1;    // a bounded mbarrier wait expired
constexpr int PGQA_DEV_BOUNDS = 2;     // bad indptr / kv_len / page id
constexpr int PGQA_DEV_CAPACITY = 4;   // work list larger than the workspace

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per wait
// Words status[kDiagFlag .. kDiagFlag + 4] after the status word: set once by the first
// wait that times out (flag, block, thread, barrier shared-memory address, parity); then,
// in that block, warp w (< 16) that leaves a wait on the abort flag writes the barrier
// address and parity it was waiting for to status[kDiagFlag + 6 + 2w], [.. + 7 + 2w].
// The status word starts a header of 64 ints; these words sit after its counters.
constexpr int kDiagFlag = 8;
constexpr int kDiagWords = 6 + 2 * 16;  // flag .. the last warp's record

// ------------------------------------------------------------------ workspace layout
// [0, 256)      header: status word, counters
// [256, 640)    three tensor maps (prefill Q, K, V), 128-byte aligned
// [1024, ...)   per-call arrays (prefill: tile offsets + work items; decode: chunk
//               offsets, sanitised kv lengths, partial results)
constexpr size_t kWsHeader = 0;
constexpr size_t kWsTmapOffset = 256;
constexpr size_t kWsArrays = 1024;
constexpr size_t kDefaultWorkspace = 128ull << 20;

struct WsHeader {
    int status;
    int n_items;      // prefill: number of work items written by the plan
    int total_q;
    int total_kv;
    int merge_rows;   // prefill: (token, head) rows the split-KV merge combines
    int pad[59];      // from word kDiagFlag on: the timeout diagnostic words
};
static_assert(sizeof(WsHeader) == 256, "workspace header size");
static_assert(kDiagFlag * sizeof(int) >= offsetof(WsHeader, pad) &&
                  (kDiagFlag + kDiagWords) * sizeof(int) <= sizeof(WsHeader),
              "the diagnostic words must not overlap the header's counters");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ prefill
namespace prefill {
constexpr int BM = 128;          // packed query rows (token x group head) per tile
constexpr int BN = 128;          // keys per K/V tile
constexpr int THREADS = 256;     // warp 0 TMA, warp 1 MMA, warps 4-7 softmax/epilogue
constexpr int PAIR_THREADS = 384;  // + warps 8-11: softmax of the second q tile
constexpr int PLAN_THREADS = 1024;
constexpr int COST_BUCKETS = 4096;
constexpr int PLAN_SMEM_BATCH = 2048;  // batches up to this size plan out of shared memory
constexpr int PLAN_STAGE_UNITS = 2048; // work lists up to this many units are staged in smem


// One work item of the prefill: a (request, kv head, first q tile, K/V chunk) plus the
// request's offsets, written by the plan kernel so the attention roles need no further
// global loads to place it.  An item covers K/V tiles [kt0, kt1) of its q tiles' range;
// part < 0: it writes the outputs; part >= 0: it writes fp32 partial results to partial
// rows part + t * Hq + h (t = token within the request), merged afterwards.
struct alignas(16) WorkItem {
    int b, g, qt, cost;
    int q_start, qo_len, kv_start, kv_len;
    int kt0, kt1, part, nch;
};

struct Params {
    const CUtensorMap* tm_q;   // in the workspace, patched by the plan kernel
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    void* o;
    float* lse;
    const int* q_indptr;
    const int* kv_indptr;
    const WorkItem* items;     // sorted longest first
    const WsHeader* hdr;
    int* status;
    int num_qo_heads;
    int num_kv_heads;
    int group;
    int causal;
    float scale_log2;          // sm_scale * log2(e) (* k_scale for a dequantised FP8 cache)
    float v_scale;             // output scale (1, or v_scale for a dequantised FP8 cache)
    int f8conv;                // K/V pages converted from E4M3: V (and so P) is f16 in P.V
    // paged K/V (paged kernels only): key j of request b is slot j % page_size of page
    // page_table[b * page_table_stride + j / page_size]; the K/V maps view each page pool
    // as a 4-D tensor {d, slot, head, page} (caller strides) with a box of one page of
    // one head and 64 columns (page_size rows)
    const int* page_table;
    int page_table_stride;
    int page_size;             // 16, 32, 64 or 128
    int num_pages;
    // grouped stage layout (head_dim 256, pages of up to 32 tokens): keys per TMA box (8,
    // or 16 when a page's (page, head) pairs can be addressed as one tensor dimension) and
    // that dimension's rows per page (page stride / head stride)
    int box_keys;
    int page_heads;
    // split-KV partial results: o [rows, D] fp32 normalised over the chunk's keys, lse
    // [rows] fp32 (natural log); merge bookkeeping from the plan
    float* part_o;
    float* part_lse;
    const int* merge_off;      // [batch + 1] first merge row of each request
    const int* part_off;       // [batch] first partial row of each request (-1: not split)
    const int* nch;            // [batch] chunks of each request
    const int* kvl;            // [batch] keys of each request
    int batch;
    int split_tiles;           // K/V tiles per chunk of a split request
};

struct PlanParams {
    const int* q_indptr;
    const int* kv_indptr;      // ragged K/V; nullptr when kv_lens is given
    const int* kv_lens;        // paged K/V: keys per request [batch]
    int max_kv;                // paged: page_table_stride * page_size
    int batch;
    int num_kv_heads;
    int group;
    int causal;
    int tiles_per_item;        // consecutive q tiles one work item covers (1 or 2)
    int split_tiles;           // K/V tiles per chunk of a split request (16 for head_dim 128,
                               // 32 for 256)
    WsHeader* hdr;
    int* tile_off;             // [batch + 1]
    int* kv_off;               // paged: [batch + 1] prefix sums of kv_lens (workspace)
    WorkItem* items;
    long long item_capacity;
    CUtensorMap* tm_out;       // 3 maps: Q, K, V
    // split-KV: allowed when split_ok; chosen when the work list would have fewer than
    // 2 * num_ctas items and the partial results fit in part_capacity rows
    int split_ok;
    int num_ctas;
    int num_qo_heads;
    long long part_capacity;
    int* unit_off;             // [batch + 1] (q item, chunk) units per request
    int* part_off;             // [batch]
    int* merge_off;            // [batch + 1]
    int* nch;                  // [batch]
    int* kvl;                  // [batch] keys per request (for the merge)
};
}  // namespace prefill

// ------------------------------------------------------------------ decode
namespace decode {
constexpr int PAGE = 16;           // tokens per TMA unit (one box); pages hold 1, 2, 4 or 8
constexpr int CHUNK = 1024;        // tokens per split-KV chunk (calls with a lot of work)
constexpr int CHUNK_MIN = 128;     // the shortest chunk
constexpr int WAVE_ITEMS = 2048;   // (request, chunk, kv head) items of about one wave of warps

// Keys per split-KV chunk, decided from the call's shape alone (batch, the page table's key
// capacity, kv heads): the longest of 1024, 512, 256, 128 keys that still gives about a
// wave of (chunk, kv head) warps, so that calls with little work spread over the GPU.  For
// a given chunk length a request's chunks depend on the request alone, so its results do
// not depend on the other requests of the batch.
// `top` caps the longest chunk: the tensor-core E4M3 decode with several query rows per
// request keeps 7 tiles of 128 keys per item (CHUNK_E4M3_ROWS), so its 1024 becomes 896.
constexpr int CHUNK_E4M3_ROWS = 896;
inline int chunk_keys(int batch, long long max_kv, int num_kv_heads, int top = CHUNK) {
    int chunk = CHUNK;
    while (chunk > CHUNK_MIN) {
        const long long per_req = max_kv > 0 ? (max_kv + chunk - 1) / chunk : 1;
        if ((long long)batch * per_req * num_kv_heads >= WAVE_ITEMS) break;
        chunk /= 2;
    }
    return chunk > top ? top : chunk;
}
inline long long total_chunks(int batch, long long max_kv, int chunk) {
    return (long long)batch * (max_kv > 0 ? (max_kv + chunk - 1) / chunk : 1);
}
constexpr int HEAD_DIM = 128;
constexpr int WARPS = 4;           // warps per CTA, one work item per warp
constexpr int STAGES = 2;          // pages in flight per warp (TMA ring in shared memory)
constexpr int PAGE_HEAD_BYTES = PAGE * HEAD_DIM * 2;               // 4 KB
constexpr int STAGE_BYTES = 2 * PAGE_HEAD_BYTES;                   // K and V of one page
constexpr int WARP_SMEM = STAGES * STAGE_BYTES + 1024;             // + scores, barriers
constexpr int SMEM_BYTES = 1024 + WARPS * WARP_SMEM;
constexpr int PLAN_THREADS = 1024;

struct Params {
    // K / V page pools as 4-D tensors {d, slot, head, page} with the caller's strides
    // (NHD, HND or a slice of a larger cache); one box is 16 slots of one head (4 KB)
    CUtensorMap tm_kpages;
    CUtensorMap tm_vpages;
    const void* q;
    const void* k_pages;
    const void* v_pages;
    const int* page_table;
    const int* kv_eff;          // sanitised kv lengths [batch]
    const int* chunk_off;       // [batch + 1]
    void* o;
    float* lse;
    float* part_o;              // [total_chunks, Hq, D]
    float* part_lse;            // [total_chunks, Hq]
    int* status;
    int batch;
    int page_table_stride;
    int page_size;              // 16, 32, 64 or 128 tokens
    int num_pages;
    int num_qo_heads;
    int num_kv_heads;
    float scale_log2;           // sm_scale * log2(e) (* k_scale for E4M3 K/V)
    float v_scale;              // output scale: 1 for bf16 K/V, v_scale for E4M3
    // query rows: request b owns rows q_off[b] .. q_off[b] + q_len[b] - 1 (sanitised by the
    // plan); q_off == nullptr: one row per request, row b (decode).  Partial results leave
    // room for max_qo rows per chunk: slot (chunk * max_qo + i) * Hq + head.
    const int* q_off;
    const int* q_len;
    int max_qo;
    int causal;
    long long chunk_capacity;
    int chunk;                  // keys per split-KV chunk (chunk_keys)
};

struct PlanParams {
    const int* kv_lens;
    int* kv_eff;
    int* chunk_off;
    int* status;
    int batch;
    int max_kv;                 // page_table_stride * page_size
    int chunk;                  // keys per split-KV chunk
    // several query rows per request (nullptr: one row per request): q_indptr [batch + 1]
    // is checked (non-decreasing, at most max_qo rows per request) into q_off / q_len
    const int* q_indptr;
    int* q_off;
    int* q_len;
    int max_qo;
};
}  // namespace decode

namespace dequant {
// E4M3 K/V pages -> a bf16 pool (dequant.cu)
struct Params {
    const uint8_t* k8;           // E4M3 pools with the caller's strides (elements = bytes)
    const uint8_t* v8;
    long long page_stride, slot_stride, head_stride;
    void* k16;                   // bf16 pools, packed NHD [pool pages][page_size][Hk][d]
    void* v16;
    const int* page_table;       // [batch][page_table_stride]
    const int* kv_lens;          // [batch]
    int* table_out;              // by table slot: [batch][page_table_stride]; by page: null
    int* status;
    int batch, page_table_stride, page_size, num_pages, num_kv_heads, head_dim;
};
}  // namespace dequant

}  // namespace pgqa
