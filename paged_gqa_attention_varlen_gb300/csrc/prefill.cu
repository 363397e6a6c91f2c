// prefill.cu -- ragged (varlen) GQA prefill attention for sm_103a.
//
// What it computes: for every request b (query rows q_indptr[b]..q_indptr[b+1]-1, key
// rows kv_indptr[b]..kv_indptr[b+1]-1), every query head h and query row i,
//   o[i,h] = softmax_j(sm_scale * q[i,h] . k[j, h/G]) v[j, h/G]   over visible keys j,
//   lse[i,h] = ln sum_j exp(sm_scale * q[i,h] . k[j, h/G]),
// with key j visible iff j < kv_len and, when causal, j <= i + kv_len - qo_len
// (bottom-right alignment).  Sources: Atlas "Module flashinfer" API page
// (ragged_prefill_bf16_hd128 / _hd256: one batched varlen launch addressed by
// q_indptr / kv_indptr); FlashInfer documentation, flashinfer_benchmark.py "Attention
// Flags" (--causal, bottom-right masking).
//
// Design (GB300-first, not the SM80 mma.sync kernel the pages describe):
//  * plan_kernel (1 CTA) validates the indptr arrays (or kv_lens for paged K/V), turns
//    them into a work list of (request, kv head, q tile(s), K/V chunk) items sorted by
//    their number of K/V tiles (longest first; records staged in shared memory and
//    written out in coalesced pieces), and patches the global extents of the TMA tensor
//    maps from q_indptr[batch] / kv_indptr[batch], so the host never reads device data.
//    Work lists too short to fill the GPU are split into request-local chunks of 2048 keys
//    (head_dim 128) or 4096 keys (head_dim 256).
//  * attention_pair_kernel (head_dim 128) is persistent (one CTA per SM) and
//    warp-specialised, two 128-row q tiles (A, B) per CTA sharing one K/V stream:
//      warp 0   TMA producer: Q tiles once per item, K/V tiles through a 4-stage ring;
//      warp 1   tcgen05.mma issuer: S_x = Q_x K^T into tensor memory, O_x += P_x V with
//               P read straight from tensor memory, alternating A and B so that one
//               tile's softmax overlaps the other tile's MMAs;
//      warps 4-11 softmax, a warpgroup per tile: one thread per packed query row (= TMEM
//               lane), masking on diagonal tiles only, online max / sum, P written back
//               as bf16 in two halves (the MMA warp starts P.V on the first), O rescaled
//               in TMEM only when the running max grows by more than 2^8; an item's
//               epilogue runs inside the next item's first tile.
//  * attention_kernel<256> (head_dim 256): one q tile per CTA, two S buffers (O alone
//    takes 256 TMEM columns), the same roles.
//  * PAGED instances read K/V through a page table: lane l of the producer warp loads
//    page l of each K/V tile as 4-D TMA boxes, and warp 2 zeroes an item's last V rows
//    past kv_len before its final P.V.
//  * merge_kernel combines split-KV partial results (fp32 O, lse) per (token, head).
//  * GQA packing: a 128-row Q tile holds 128/G tokens x the G query heads that share a
//    KV head (3-D TMA box), so each K/V tile is read once for all G heads.
#include <atomic>

#include "ptx.cuh"

namespace pgqa {
namespace prefill {

struct Geo {
    int q_start, qo_len, kv_start, kv_len;
    int t0;          // first token (within the request) of the item's q tile
    int n_tiles;     // K/V tiles with at least one visible key for some row of the tile
    int n_unmasked;  // leading tiles in which every row sees every key
};

__device__ __forceinline__ Geo tile_geometry(int q_start, int qo_len, int kv_start, int kv_len,
                                             int qt, int group, int causal) {
    Geo x;
    x.q_start = q_start;
    x.qo_len = qo_len;
    x.kv_start = kv_start;
    x.kv_len = kv_len;
    const int tpt = BM / group;
    x.t0 = qt * tpt;
    const int t1 = min(x.qo_len, x.t0 + tpt);
    int n_keys = x.kv_len;
    if (causal) n_keys = max(0, min(x.kv_len, t1 + x.kv_len - x.qo_len));
    x.n_tiles = (n_keys + BN - 1) / BN;
    const int lim = causal ? min(x.t0 + x.kv_len - x.qo_len, x.kv_len - 1) : x.kv_len - 1;
    x.n_unmasked = lim >= 0 ? min((lim + 1) / BN, x.n_tiles) : 0;
    return x;
}

__device__ __forceinline__ Geo item_geometry(const int* q_indptr, const int* kv_indptr, int b,
                                             int qt, int group, int causal) {
    return tile_geometry(q_indptr[b], q_indptr[b + 1] - q_indptr[b], kv_indptr[b],
                         kv_indptr[b + 1] - kv_indptr[b], qt, group, causal);
}

// geometry of q tile (w.qt + dt) of a work item
__device__ __forceinline__ Geo geo_of(const WorkItem& w, int dt, int group, int causal) {
    return tile_geometry(w.q_start, w.qo_len, w.kv_start, w.kv_len, w.qt + dt, group, causal);
}

// The attention kernels start while the plan still writes the work list (programmatic
// dependent launch), so it is read through L2 (ld.global.cg), never through the
// non-coherent read-only path, whose contract is data that no one writes while the
// kernel runs.
__device__ __forceinline__ WorkItem load_item(const WorkItem* items, int i) {
    const int4* v = reinterpret_cast<const int4*>(items + i);
    const int4 a = __ldcg(v), c = __ldcg(v + 1), e = __ldcg(v + 2);
    WorkItem w;
    w.b = a.x; w.g = a.y; w.qt = a.z; w.cost = a.w;
    w.q_start = c.x; w.qo_len = c.y; w.kv_start = c.z; w.kv_len = c.w;
    w.kt0 = e.x; w.kt1 = e.y; w.part = e.z; w.nch = e.w;
    return w;
}

// K/V chunks of a request of kv_len keys when its work is split into chunks of st tiles
__host__ __device__ __forceinline__ int split_chunks(int kv_len, int st) {
    const int tiles = (kv_len + BN - 1) / BN;
    return tiles > st ? (tiles + st - 1) / st : 1;
}


// Items are sorted longest first; CTA c walks them in "snake" order (rounds of gridDim
// items, alternate rounds reversed), which balances the per-CTA totals of an LPT-sorted
// list far better than a plain stride.  Every role of a CTA walks the same sequence.
__device__ __forceinline__ int snake_next(int& r, int n) {
    const int ncta = gridDim.x, cta = blockIdx.x;
    for (;;) {
        ++r;
        if ((long long)r * ncta >= n) return -1;
        const int idx = r * ncta + ((r & 1) ? ncta - 1 - cta : cta);
        if (idx < n) return idx;
    }
}

__device__ __forceinline__ int find_segment(const int* off, int n, int f) {
    // largest b in [0, n) with off[b] <= f
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= f) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// K/V tiles of the longest q tile of an item (the item covers tiles qt..qt+tpi-1 that exist)
__device__ __forceinline__ int item_cost(const PlanParams& p, const int* qi, const int* ki, int b,
                                         int qt) {
    const long long qo = qi[b + 1] - qi[b];
    const int tiles = (int)((qo * p.group + BM - 1) / BM);
    const int last = min(qt + p.tiles_per_item, tiles) - 1;
    return item_geometry(qi, ki, b, last, p.group, p.causal).n_tiles;
}

// Block-wide inclusive scan of one int per thread (blockDim.x == PLAN_THREADS): warp
// shuffles, then a scan of the 32 warp totals.  `wsum` is 32 ints of shared memory.
// Returns the inclusive prefix; *total receives the block total.
__device__ __forceinline__ int block_inclusive_scan(int v, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? wsum[warp - 1] : 0);
    *total = wsum[31];
    __syncthreads();  // wsum may be reused by the next call
    return r;
}

// ---------------------------------------------------------------------------- plan
__global__ void __launch_bounds__(PLAN_THREADS)
    plan_kernel(PlanParams p, const __grid_constant__ CUtensorMap tq,
                const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    // the attention kernel may launch now; it waits for this grid before reading the plan
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int hist[COST_BUCKETS];
    __shared__ int scan[PLAN_THREADS];
    __shared__ alignas(128) CUtensorMap smap[3];
    // batches up to PLAN_SMEM_BATCH keep indptr and the per-request item offsets in shared
    // memory, so the binary searches below do not wait on L2
    __shared__ int s_qi[PLAN_SMEM_BATCH + 1], s_ki[PLAN_SMEM_BATCH + 1],
        s_off[PLAN_SMEM_BATCH + 1];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const bool small = p.batch <= PLAN_SMEM_BATCH;
    const bool paged = p.kv_lens != nullptr;
    if (small) {
        for (int b = tid; b <= p.batch; b += nthr) {
            s_qi[b] = p.q_indptr[b];
            if (!paged) s_ki[b] = p.kv_indptr[b];
        }
        __syncthreads();
    }
    const int* qi = small ? s_qi : p.q_indptr;
    const int* ki = small ? s_ki : p.kv_indptr;
    int* toff = small ? s_off : p.tile_off;

    int bad = 0;
    if (paged) {
        // keys per request from kv_lens (0 <= kv_len <= page_table_stride * page_size),
        // turned into offsets so the rest of the plan reads them like kv_indptr; only
        // differences of these offsets are used, so unsigned wrap-around is harmless
        int* kvp = small ? s_ki : p.kv_off;
        unsigned running = 0;
        for (int base = 0; base < p.batch; base += nthr) {
            const int b = base + tid;
            int n = 0;
            if (b < p.batch) {
                n = p.kv_lens[b];
                if (n < 0 || n > p.max_kv) {
                    bad = 1;
                    n = 0;
                }
            }
            int tot;
            const int inc = block_inclusive_scan(n, scan, &tot);
            if (b < p.batch) kvp[b + 1] = (int)(running + (unsigned)inc);
            running += (unsigned)tot;
        }
        if (tid == 0) kvp[0] = 0;
        __syncthreads();
        ki = kvp;
    }
    for (int b = tid; b < p.batch; b += nthr) {
        const int q0 = qi[b], q1 = qi[b + 1];
        if (q0 < 0 || q1 < q0) bad = 1;
        if (!paged) {
            const int k0 = ki[b], k1 = ki[b + 1];
            if (k0 < 0 || k1 < k0) bad = 1;
        }
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            atomicOr(&p.hdr->status, PGQA_DEV_BOUNDS);
            p.hdr->n_items = 0;
            p.hdr->merge_rows = 0;  // the merge kernel must not run on a stale count
        }
        return;
    }

    // exclusive scan of per-request item counts -> toff
    int running = 0;
    for (int base = 0; base < p.batch; base += nthr) {
        const int b = base + tid;
        int cnt = 0;
        if (b < p.batch) {
            const long long qo = qi[b + 1] - qi[b];
            const int tiles = (int)((qo * p.group + BM - 1) / BM);
            cnt = (tiles + p.tiles_per_item - 1) / p.tiles_per_item;
        }
        int tot;
        const int inc = block_inclusive_scan(cnt, scan, &tot);
        if (b < p.batch) toff[b] = running + inc - cnt;
        running += tot;
    }
    const int total_tiles = running;
    if (tid == 0) toff[p.batch] = total_tiles;

    // Split-KV: a work list too short to fill the grid (decode-like calls: few requests,
    // few query rows, long keys) has its requests cut into chunks of split_tiles K/V tiles
    // (2048 keys for head_dim 128, 4096 for 256: measured on short hd256 lists, the longer
    // chunks halve the per-item start-up that each chunk pays).
    // The cut depends on the request alone, so within this regime a request's results do
    // not depend on the batch.  Units are (q item, chunk); chunked requests write fp32
    // partial results that the merge kernel combines.  If the partial results would not
    // fit in the workspace the work is not split.
    bool split = p.split_ok && (long long)total_tiles * p.num_kv_heads < 2LL * p.num_ctas;
    long long part_total = 0;
    int merge_total = 0, unit_total = total_tiles;
    if (split) {
        int unit_run = 0, merge_run = 0;
        for (int base = 0; base < p.batch; base += nthr) {
            const int b = base + tid;
            int units = 0, prow = 0, mrow = 0, nc = 1;
            if (b < p.batch) {
                const int qo = qi[b + 1] - qi[b];
                const int tiles = (int)(((long long)qo * p.group + BM - 1) / BM);
                const int qitems = (tiles + p.tiles_per_item - 1) / p.tiles_per_item;
                nc = qo > 0 ? split_chunks(ki[b + 1] - ki[b], p.split_tiles) : 1;
                units = qitems * nc;
                if (nc > 1) {
                    prow = nc * qo * p.num_qo_heads;
                    mrow = qo * p.num_qo_heads;
                }
            }
            int tot_u, tot_p, tot_m;
            const int inc_u = block_inclusive_scan(units, scan, &tot_u);
            const int inc_p = block_inclusive_scan(prow, scan, &tot_p);
            const int inc_m = block_inclusive_scan(mrow, scan, &tot_m);
            if (b < p.batch) {
                p.unit_off[b] = unit_run + inc_u - units;
                p.part_off[b] = nc > 1 ? (int)(part_total + inc_p - prow) : -1;
                p.merge_off[b] = merge_run + inc_m - mrow;
                p.nch[b] = nc;
                p.kvl[b] = ki[b + 1] - ki[b];
            }
            unit_run += tot_u;
            part_total += tot_p;
            merge_run += tot_m;
        }
        if (tid == 0) {
            p.unit_off[p.batch] = unit_run;
            p.merge_off[p.batch] = merge_run;
        }
        unit_total = unit_run;
        merge_total = merge_run;
        // the same in every thread: the split list must fit where the unsplit one would
        if (part_total > p.part_capacity ||
            (long long)unit_total * p.num_kv_heads > p.item_capacity)
            split = false;
        __syncthreads();
    }
    if (!split) {
        unit_total = total_tiles;
        merge_total = 0;
    }
    const int* uoff = split ? p.unit_off : toff;
    const long long n_items = (long long)unit_total * p.num_kv_heads;
    if (n_items > p.item_capacity) {
        if (tid == 0) {
            atomicOr(&p.hdr->status, PGQA_DEV_CAPACITY);
            p.hdr->n_items = 0;
            p.hdr->merge_rows = 0;
        }
        return;
    }
    for (int i = tid; i < COST_BUCKETS; i += nthr) hist[i] = 0;
    __syncthreads();

    // a unit: request b, q item qt, chunk c (0 when not split) and its K/V-tile cost
    auto unit_of = [&](int f, int& b, int& qt, int& c, int& cost) {
        b = find_segment(uoff, p.batch, f);
        const int local = f - uoff[b];
        const int nc = split ? p.nch[b] : 1;
        qt = (local / nc) * p.tiles_per_item;
        c = local % nc;
        const int full = item_cost(p, qi, ki, b, qt);
        cost = nc > 1 ? max(0, min(full - c * p.split_tiles, p.split_tiles)) : full;
    };

    // histogram of unit costs (K/V tiles of the unit's longest q tile)
    for (int f = tid; f < unit_total; f += nthr) {
        int b, qt, c, cost;
        unit_of(f, b, qt, c, cost);
        atomicAdd(&hist[min(cost, COST_BUCKETS - 1)], 1);
    }
    __syncthreads();

    // descending exclusive scan: start[c] = number of items with a larger cost
    constexpr int PER = COST_BUCKETS / PLAN_THREADS;
    int local[PER];
    int sum = 0;
    if (tid < COST_BUCKETS / PER) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            local[e] = hist[COST_BUCKETS - 1 - (tid * PER + e)];
            sum += local[e];
        }
    }
    int tot;
    const int inc = block_inclusive_scan(sum, scan, &tot);
    if (tid < COST_BUCKETS / PER) {
        int acc = inc - sum;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            hist[COST_BUCKETS - 1 - (tid * PER + e)] = acc;
            acc += local[e];
        }
    }
    __syncthreads();

    // scatter: the kv heads of one unit take consecutive slots.  With up to
    // PLAN_STAGE_UNITS units each unit's record goes to shared memory at its sorted slot,
    // and the whole list is then written out in consecutive 16-byte pieces; longer lists
    // write each unit's kv-head items directly.
    extern __shared__ __align__(16) uint8_t plan_dyn[];
    WorkItem* staged = reinterpret_cast<WorkItem*>(plan_dyn);
    const bool stage = unit_total <= PLAN_STAGE_UNITS;
    for (int f = tid; f < unit_total; f += nthr) {
        int b, qt, c, cost;
        unit_of(f, b, qt, c, cost);
        const int slot = atomicAdd(&hist[min(cost, COST_BUCKETS - 1)], 1);
        const int q0 = qi[b], k0 = ki[b];
        const int nc = split ? p.nch[b] : 1;
        WorkItem w;
        w.b = b;
        w.qt = qt;
        w.cost = cost;
        w.q_start = q0;
        w.qo_len = qi[b + 1] - q0;
        w.kv_start = k0;
        w.kv_len = ki[b + 1] - k0;
        w.kt0 = nc > 1 ? c * p.split_tiles : 0;
        w.kt1 = nc > 1 ? (c + 1) * p.split_tiles : 0x7fffffff;
        w.part = nc > 1 ? p.part_off[b] + c * w.qo_len * p.num_qo_heads : -1;
        w.nch = nc;
        if (stage) {
            w.g = 0;
            staged[slot] = w;
        } else {
            for (int g = 0; g < p.num_kv_heads; ++g) {
                w.g = g;
                p.items[(long long)slot * p.num_kv_heads + g] = w;
            }
        }
    }
    if (stage) {
        __syncthreads();
        constexpr int PIECES = (int)(sizeof(WorkItem) / sizeof(int4));  // 16-byte pieces
        const int hk = p.num_kv_heads;
        const int4* src = reinterpret_cast<const int4*>(staged);
        int4* dst = reinterpret_cast<int4*>(p.items);
        for (int i = tid; i < (int)n_items * PIECES; i += nthr) {
            const int item = i / PIECES, piece = i - item * PIECES;
            const int u = item / hk;
            int4 v = src[u * PIECES + piece];
            if (piece == 0) v.y = item - u * hk;  // WorkItem::g
            dst[i] = v;
        }
    }

    // tensor maps with the real row extents
    if (tid < 32) {
        const int total_q = qi[p.batch];
        const int total_kv = ki[p.batch];
        if (tid == 0) {
            smap[0] = tq;
            smap[1] = tk;
            smap[2] = tv;
            tensormap_set_dim_smem<2>(smem_u32(&smap[0]), (uint32_t)max(total_q, 1));
            if (!paged) {  // paged maps span the page pool, whose size the host knows
                tensormap_set_dim_smem<1>(smem_u32(&smap[1]), (uint32_t)max(total_kv, 1));
                tensormap_set_dim_smem<1>(smem_u32(&smap[2]), (uint32_t)max(total_kv, 1));
            }
            p.hdr->n_items = (int)n_items;
            p.hdr->total_q = total_q;
            p.hdr->total_kv = total_kv;
            p.hdr->merge_rows = merge_total;
        }
        __syncwarp();
        tensormap_publish(p.tm_out + 0, smem_u32(&smap[0]));
        tensormap_publish(p.tm_out + 1, smem_u32(&smap[1]));
        tensormap_publish(p.tm_out + 2, smem_u32(&smap[2]));
    }
}

// ------------------------------------------------------------------ paged K/V
// With paged K/V the producer is a whole warp: lane l owns page l of a K/V tile (a tile
// of BN keys spans BN / page_size pages).  Pages past a request's last key are never read.
// Page id of lane l for tile j (-1 if that page holds no key of the request).
__device__ __forceinline__ int lane_page_id(const int* pt_row, int j, int ppt, int npg, int lane) {
    const int pg = j * ppt + lane;
    return lane < ppt && pg < npg ? __ldcg(pt_row + pg) : -1;  // see load_item
}
// Whether lane l's page of tile j is in use, reporting an id outside the page pool
// (PGQA_DEV_BOUNDS; that page is then not loaded).
__device__ __forceinline__ bool lane_page_ok(int id, int j, int ppt, int npg, int num_pages,
                                             int lane, int* status) {
    const bool in_use = lane < ppt && j * ppt + lane < npg;
    const bool ok = in_use && id >= 0 && id < num_pages;
    if (in_use && !ok) atomicOr(status, PGQA_DEV_BOUNDS);
    return ok;
}
// Warp-collective: arm `bar` with the bytes of every valid page box of this load (lane 0),
// then each lane issues the boxes of its own page(s) of kv head g: one box per 64-column
// chunk, landing at rows lane * ps .. of every chunk of the stage, the layout a single
// 128-row box would have written.  The maps are 4-D {d, slot, head, page}.
template <int CHUNKS, int CHUNK_BYTES>
__device__ __forceinline__ void issue_page_boxes(uint32_t bar, int ps, int g, int lane,
                                                 bool v_ok, uint32_t v_dst, const CUtensorMap* tm_v,
                                                 int v_id, bool k_ok, uint32_t k_dst,
                                                 const CUtensorMap* tm_k, int k_id) {
    const int n = __popc(__ballot_sync(0xffffffffu, v_ok)) +
                  __popc(__ballot_sync(0xffffffffu, k_ok));
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(n * CHUNKS * ps * 128));
    __syncwarp();
    const uint32_t row_off = (uint32_t)(lane * ps * 128);
    if (v_ok) {
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c)
            tma_load_4d(v_dst + c * CHUNK_BYTES + row_off, tm_v, bar, c * 64, 0, g, v_id);
    }
    if (k_ok) {
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c)
            tma_load_4d(k_dst + c * CHUNK_BYTES + row_off, tm_k, bar, c * 64, 0, g, k_id);
    }
}

// Zero rows r0..BM-1 of every chunk of a K/V stage (warp-collective).  With the 128-byte
// swizzle each row's 128 bytes stay within its own 128-byte line, so whole lines are
// cleared.  The writes are then fenced for the tensor core's async-proxy reads.
template <int CHUNKS, int CHUNK_BYTES>
__device__ __forceinline__ void zero_stage_rows(uint32_t stage, int r0, int lane) {
    const int n16 = (BM - r0) * 8;  // 16-byte units per chunk
    for (int c = 0; c < CHUNKS; ++c) {
        const uint32_t base = stage + c * CHUNK_BYTES + r0 * 128;
        for (int u = lane; u < n16; u += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + u * 16), "r"(0)
                         : "memory");
    }
    fence_async_smem();
}

// Grouped stage layout (paged K/V with small pages, head_dim 256): a 128-key stage is 16
// groups of 8 keys, group i at i * (D / 64) KB, and within a group the 64-column chunks
// (one 128-byte swizzle atom of 8 rows each) 1 KB apart.  A TMA box of a 5-D map fills
// one or two consecutive groups, all chunks: with box_keys = 16 the map is {64 columns,
// 8 slots, chunk, 8-slot half of a page, (page, head)} and a box is 16 slots of one page
// and head; with box_keys = 8 (page and head kept as separate dimensions) it is
// {64 columns, slot, chunk, head, page} and a box is 8 slots.  A 64 KB tile of 16-token
// pages is then 8 (or 16) boxes instead of 32 boxes of 2 KB; the tensor core reads the
// same swizzle atoms, with 8-row groups (D / 64) KB apart instead of 1 KB.
// Lane l < 128 / box_keys of the producer warp loads box l of tile j: keys
// box_keys * l .. + box_keys - 1 of the tile, in page (j * 128 + box_keys * l) / page_size.
__device__ __forceinline__ int group_page_id(const int* pt_row, int j, int ps, int npg, int bk,
                                             int lane) {
    const int pg = (j * BN + bk * lane) / ps;
    return lane < BN / bk && pg < npg ? __ldcg(pt_row + pg) : -1;  // see load_item
}
__device__ __forceinline__ bool group_page_ok(int id, int j, int ps, int npg, int bk,
                                              int num_pages, int lane, int* status) {
    const bool in_use = lane < BN / bk && (j * BN + bk * lane) / ps < npg;
    const bool ok = in_use && id >= 0 && id < num_pages;
    if (in_use && !ok) atomicOr(status, PGQA_DEV_BOUNDS);
    return ok;
}
// Warp-collective: lane 0 arms `bar` with the bytes of every valid box, then each lane with
// a valid page loads its box of kv head g.
template <int GROUP_BYTES>
__device__ __forceinline__ void issue_group_boxes(uint32_t bar, int ps, int g, int bk,
                                                  int page_heads, int lane, bool ok, uint32_t dst,
                                                  const CUtensorMap* tm, int id) {
    const int n = __popc(__ballot_sync(0xffffffffu, ok));
    const int box_bytes = GROUP_BYTES * (bk / 8);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(n * box_bytes));
    __syncwarp();
    if (ok) {
        const int slot = (bk * lane) % ps;
        if (bk == 16)
            tma_load_5d(dst + lane * box_bytes, tm, bar, 0, 0, 0, slot / 8, id * page_heads + g);
        else
            tma_load_5d(dst + lane * box_bytes, tm, bar, 0, slot, 0, g, id);
    }
}
// Zero rows r0..BN-1 of a grouped stage (warp-collective): whole 128-byte lines, fenced for
// the tensor core's async-proxy reads.
template <int CHUNKS>
__device__ __forceinline__ void zero_group_rows(uint32_t stage, int r0, int lane) {
    const int n16 = (BN - r0) * CHUNKS * 8;  // 16-byte units
    for (int u = lane; u < n16; u += 32) {
        const int r = r0 + u / (CHUNKS * 8), rest = u % (CHUNKS * 8);
        const uint32_t a = stage + (r >> 3) * (CHUNKS * 1024) + (rest >> 3) * 1024 + (r & 7) * 128 +
                           (rest & 7) * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
    }
    fence_async_smem();
}

// ---------------------------------------------------------------------- attention
template <int D>
struct Cfg {
    static constexpr int CHUNKS = D / 64;              // 64-element (128-byte) swizzle chunks
    static constexpr int CHUNK_BYTES = BM * 128;       // one chunk of a 128-row tile
    static constexpr int TILE_BYTES = BM * D * 2;      // Q tile = K tile = V tile
    static constexpr int STAGES = D == 128 ? 4 : 2;
    static constexpr int TMEM_O = 256;                 // S buffers at columns 0 and 128
    static constexpr int TMEM_COLS = 512;
    static constexpr int NUM_BARS = 2 + 2 * STAGES + 10;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES * (1 + STAGES) + 8 * NUM_BARS + 16;
};

// Growth of the running max (log2 units) below which O and l keep their old scale:
// probabilities then stay below 2^8 and the fp32 accumulators are unaffected, while the
// O rescale in tensor memory is skipped for most tiles.
constexpr float kRescaleThreshold = 8.0f;

// K/V tiles this item covers for a q tile of geometry x: [kt0, kt0 + n)
__device__ __forceinline__ int item_tiles(const WorkItem& w, const Geo& x) {
    return max(0, min(w.kt1, x.n_tiles) - w.kt0);
}

// The wait on tcgen05.ld results names the destination registers, so no use of them can
// be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
          "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
          "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
          "+r"(r[31])
        :
        : "memory");
}

// F8CONV: K/V pages converted from an E4M3 cache, V to f16: P is rounded to f16 (not bf16)
// and P.V runs on f16 operands, which keeps 11 bits of each weight instead of 8.
template <int D, bool PAGED, bool GROUPED, bool F8CONV>
__global__ void __launch_bounds__(THREADS, 1) attention_kernel(const Params p) {
    using C = Cfg<D>;
    static_assert(!GROUPED || PAGED, "the grouped layout is for paged K/V");
    static_assert(!F8CONV || PAGED, "converted pages are paged");
    // K/V stage layout: byte stride between 64-column chunks and between 8-row groups
    constexpr uint32_t KV_CH = GROUPED ? 1024u : (uint32_t)C::CHUNK_BYTES;
    constexpr uint32_t KV_SBO = GROUPED ? (uint32_t)C::CHUNKS * 1024u : 1024u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::TILE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE_BYTES * (1 + C::STAGES));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    const int Q_FULL = 0, Q_EMPTY = 1, KV_FULL = 2, KV_EMPTY = 2 + C::STAGES;
    // FIX_READY / V_FIXED: paged K/V only, as in the two-tile kernel (warp 2 zeroes the
    // rows past kv_len of an item's last V tile before its P.V).
    // PV_DONE completes after every P.V; the softmax waits on it only before rescaling O
    // (when S_FULL of tile t has fired, the P.V of tile t - 2 is done and that of tile t
    // cannot start, so PV_DONE is at most one phase from tile t - 1's: a parity wait is
    // exact even though most tiles skip it).  PV_LAST completes once per item, after its
    // last P.V: the epilogue waits on it.
    const int S_FULL = 2 + 2 * C::STAGES, P_FULL = S_FULL + 2, PV_DONE = P_FULL + 2,
              O_EMPTY = PV_DONE + 1, MMA_DRAIN = O_EMPTY + 1, FIX_READY = MMA_DRAIN + 1,
              V_FIXED = FIX_READY + 1, PV_LAST = V_FIXED + 1;
    static_assert(PV_LAST + 1 == C::NUM_BARS, "barrier count");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(BAR(Q_FULL), 1);
        mbar_init(BAR(Q_EMPTY), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(BAR(KV_FULL + s), 1);
            mbar_init(BAR(KV_EMPTY + s), 1);
        }
        mbar_init(BAR(S_FULL), 1);
        mbar_init(BAR(S_FULL + 1), 1);
        mbar_init(BAR(P_FULL), 128);
        mbar_init(BAR(P_FULL + 1), 128);
        mbar_init(BAR(PV_DONE), 1);
        mbar_init(BAR(O_EMPTY), 128);
        mbar_init(BAR(MMA_DRAIN), 1);
        mbar_init(BAR(FIX_READY), 1);
        mbar_init(BAR(V_FIXED), 32);
        mbar_init(BAR(PV_LAST), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the prologue above overlapped the plan kernel; its outputs are read from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem_base = *tmem_slot;

    const int n_items = __ldcg(&p.hdr->n_items);  // written by the plan
    const int G = p.group;

    if (warp == 0 || (PAGED && warp == 3)) {
        // ------------------------------------------------------------ TMA producer
        // Ragged K/V: lane 0 alone.  Paged K/V: the whole warp, lane l loading page l of
        // each K/V tile (its id read one load ahead); lane 0 arms the barriers.  Paged:
        // warps 0 and 3 take alternate loads (the ring positions load_idx % 2), so two
        // warps issue boxes; both follow the page ids of every tile.
        constexpr uint32_t NPROD = PAGED ? 2u : 1u;
        const uint32_t pw = warp == 0 ? 0u : 1u;
        if (PAGED || lane == 0) {
            auto wait = [&](uint32_t bar, uint32_t par) -> bool {
                if constexpr (PAGED)
                    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, par, abort_flag, p.status));
                else
                    return mbar_wait_bounded(bar, par, abort_flag, p.status);
            };
            tensormap_acquire(p.tm_q);
            tensormap_acquire(p.tm_k);
            tensormap_acquire(p.tm_v);
            const int ps = p.page_size;
            const int ppt = PAGED ? BN / ps : 0;
            uint32_t load_idx = 0, q_count = 0;
            bool ok = true;
            int rr = -1;
            int it = snake_next(rr, n_items);
            while (ok && it >= 0) {
                const WorkItem w = load_item(p.items, it);
                it = snake_next(rr, n_items);
                const Geo x = geo_of(w, 0, G, p.causal);
                const int n = item_tiles(w, x);  // K/V tiles kt0 .. kt0 + n - 1
                const int kt0 = w.kt0;
                if (n == 0) continue;
                if (pw == 0) {
                    ok = wait(BAR(Q_EMPTY), (q_count & 1) ^ 1);
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(BAR(Q_FULL), C::TILE_BYTES);
#pragma unroll
                        for (int c = 0; c < C::CHUNKS; ++c)
                            tma_load_3d(sQ + c * C::CHUNK_BYTES, p.tm_q, BAR(Q_FULL), c * 64,
                                        w.g * G, x.q_start + x.t0);
                    }
                    ++q_count;
                }
                // consumption order of the MMA warp: K0, (K1, V0), (K2, V1), ..., V_{n-1}
                // (tile indices relative to kt0)
                const int nl = 2 * n;
                auto tile_of = [&](int s, bool& is_k) -> int {
                    if (s == 0) {
                        is_k = true;
                        return 0;
                    }
                    if (s == nl - 1) {
                        is_k = false;
                        return n - 1;
                    }
                    const int pr = (s - 1) >> 1;
                    is_k = ((s - 1) & 1) == 0;
                    return is_k ? pr + 1 : pr;
                };
                const int* pt_row = PAGED ? p.page_table + (size_t)w.b * p.page_table_stride : nullptr;
                const int npg = PAGED ? (x.kv_len + ps - 1) / ps : 0;
                // paged: K_j and V_j share tile j's pages.  This lane's page ids of the
                // last two K tiles issued (V loads reuse them) and of the next K tile,
                // whose read is started one K load ahead.
                auto page_id = [&](int jj) -> int {
                    if constexpr (GROUPED)
                        return group_page_id(pt_row, jj, ps, npg, p.box_keys, lane);
                    else return lane_page_id(pt_row, jj, ppt, npg, lane);
                };
                int id_next = PAGED ? page_id(kt0) : -1;
                int id_last = -1, id_prev = -1, k_last = -1;
                for (int s = 0; s < nl; ++s) {
                    bool is_k;
                    const int jr = tile_of(s, is_k);
                    const int j = kt0 + jr;  // absolute K/V tile of the request
                    const uint32_t st = load_idx % C::STAGES;
                    const CUtensorMap* tm = is_k ? p.tm_k : p.tm_v;
                    if constexpr (PAGED) {
                        int pid;
                        if (is_k) {
                            pid = id_next;
                            id_prev = id_last;
                            id_last = id_next;
                            k_last = j;
                            if (jr + 1 < n) id_next = page_id(j + 1);
                        } else {
                            pid = j == k_last ? id_last : id_prev;
                        }
                        if (load_idx % NPROD != pw) {  // the other producer's load
                            ++load_idx;
                            continue;
                        }
                        ok = wait(BAR(KV_EMPTY + st), ((load_idx / C::STAGES) & 1) ^ 1);
                        if (!ok) break;
                        if constexpr (GROUPED) {
                            const bool pg_ok = group_page_ok(pid, j, ps, npg, p.box_keys,
                                                             p.num_pages, lane, p.status);
                            issue_group_boxes<(int)KV_SBO>(BAR(KV_FULL + st), ps, w.g, p.box_keys,
                                                           p.page_heads, lane, pg_ok,
                                                           sKV + st * C::TILE_BYTES, tm, pid);
                        } else {
                            const bool pg_ok = lane_page_ok(pid, j, ppt, npg, p.num_pages, lane,
                                                            p.status);
                            issue_page_boxes<C::CHUNKS, C::CHUNK_BYTES>(
                                BAR(KV_FULL + st), ps, w.g, lane, false, 0, tm, 0, pg_ok,
                                sKV + st * C::TILE_BYTES, tm, pid);
                        }
                        if (lane == 0 && s == nl - 1 && (kt0 + n) * BN > x.kv_len)
                            mbar_arrive(BAR(FIX_READY));
                    } else {
                        ok = wait(BAR(KV_EMPTY + st), ((load_idx / C::STAGES) & 1) ^ 1);
                        if (!ok) break;
                        mbar_arrive_expect_tx(BAR(KV_FULL + st), C::TILE_BYTES);
#pragma unroll
                        for (int c = 0; c < C::CHUNKS; ++c)
                            tma_load_2d(sKV + st * C::TILE_BYTES + c * C::CHUNK_BYTES, tm,
                                        BAR(KV_FULL + st), w.g * D + c * 64, x.kv_start + j * BN);
                    }
                    ++load_idx;
                }
            }
            if (!ok && lane == 0) {
                // let every copy this warp issued land before the CTA exits
                const uint32_t first = load_idx > (uint32_t)C::STAGES ? load_idx - C::STAGES : 0;
                for (uint32_t k = first; k < load_idx; ++k)
                    if (k % NPROD == pw)
                        mbar_wait_bounded(BAR(KV_FULL + k % C::STAGES), (k / C::STAGES) & 1,
                                          nullptr, p.status);
                if (pw == 0 && q_count > 0)
                    mbar_wait_bounded(BAR(Q_FULL), (q_count - 1) & 1, nullptr, p.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t IDESC_PV =
                F8CONV ? idesc_f16_f32(BM, D, true) : idesc_bf16_f32(BM, D, true);
            uint32_t load_idx = 0, q_count = 0, tile_ctr = 0, item_cnt = 0, fixes = 0;
            bool ok = true;
            auto issue_pv = [&](int jj, int n, bool fix) -> bool {
                const uint32_t ctr = tile_ctr + jj;
                if (!mbar_wait_bounded(BAR(P_FULL + (ctr & 1)), (ctr >> 1) & 1, abort_flag,
                                       p.status))
                    return false;
                const uint32_t st = load_idx % C::STAGES;
                if (fix && jj == n - 1) {  // the last V tile, its tail rows zeroed
                    if (!mbar_wait_bounded(BAR(V_FIXED), fixes & 1, abort_flag, p.status))
                        return false;
                    ++fixes;
                } else if (!mbar_wait_bounded(BAR(KV_FULL + st), (load_idx / C::STAGES) & 1,
                                              abort_flag, p.status)) {
                    return false;
                }
                ++load_idx;
                if (jj == 0 && item_cnt > 0 &&
                    !mbar_wait_bounded(BAR(O_EMPTY), (item_cnt - 1) & 1, abort_flag, p.status))
                    return false;
                tc_fence_after();
                const uint32_t p_col = (ctr & 1) ? 128u : 0u;
                // V tile, MN-major: 16 keys = two 8-row swizzle groups (KV_SBO apart);
                // consecutive 64-column chunks of the head dim are KV_CH apart.
                // A descriptor's address field is addr / 16, so offsets add to it directly.
                const uint64_t vdesc = sdesc_sw128(sKV + st * C::TILE_BYTES, KV_CH, KV_SBO);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ts(tmem_base + C::TMEM_O, tmem_base + p_col + k * 8,
                           vdesc + (uint64_t)(k * 2 * KV_SBO / 16), IDESC_PV,
                           (jj > 0 || k > 0) ? 1u : 0u);
                mma_commit(BAR(KV_EMPTY + st));
                mma_commit(BAR(PV_DONE));
                if (jj == n - 1) mma_commit(BAR(PV_LAST));
                return true;
            };
            int rr = -1;
            int it = snake_next(rr, n_items);
            while (ok && it >= 0) {
                const WorkItem w = load_item(p.items, it);
                it = snake_next(rr, n_items);
                const Geo x = geo_of(w, 0, G, p.causal);
                const int n = item_tiles(w, x);
                if (n == 0) continue;
                const bool fix = PAGED && (w.kt0 + n) * BN > x.kv_len;
                ok = mbar_wait_bounded(BAR(Q_FULL), q_count & 1, abort_flag, p.status);
                ++q_count;
                if (!ok) break;
                tc_fence_after();
                for (int j = 0; j < n; ++j) {
                    const uint32_t st = load_idx % C::STAGES;
                    ok = mbar_wait_bounded(BAR(KV_FULL + st), (load_idx / C::STAGES) & 1,
                                           abort_flag, p.status);
                    if (!ok) break;
                    ++load_idx;
                    tc_fence_after();
                    const uint32_t ctr = tile_ctr + j;
                    const uint32_t s_col = (ctr & 1) ? 128u : 0u;
                    const uint64_t kdesc = sdesc_sw128(sKV + st * C::TILE_BYTES, 16, KV_SBO);
                    const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t qoff = ((k >> 2) * C::CHUNK_BYTES + (k & 3) * 32) / 16;
                        const uint64_t koff = ((k >> 2) * KV_CH + (k & 3) * 32) / 16;
                        mma_ss(tmem_base + s_col, qdesc + qoff, kdesc + koff, IDESC_QK,
                               k > 0 ? 1u : 0u);
                    }
                    mma_commit(BAR(KV_EMPTY + st));
                    mma_commit(BAR(S_FULL + (ctr & 1)));
                    if (j == n - 1) mma_commit(BAR(Q_EMPTY));
                    if (j >= 1) {
                        ok = issue_pv(j - 1, n, fix);
                        if (!ok) break;
                    }
                }
                if (ok) ok = issue_pv(n - 1, n, fix);
                tile_ctr += n;
                ++item_cnt;
            }
            // every MMA issued has completed before tensor memory is released
            mma_commit(BAR(MMA_DRAIN));
            mbar_wait_bounded(BAR(MMA_DRAIN), 0, nullptr, p.status);
        }
    } else if (PAGED && warp == 2) {
        // ------------------------------------------------------------ V tail fixer
        uint32_t load_idx = 0, fixes = 0;
        bool ok = true;
        int rr = -1;
        int it = snake_next(rr, n_items);
        while (ok && it >= 0) {
            const WorkItem w = load_item(p.items, it);
            it = snake_next(rr, n_items);
            const Geo x = geo_of(w, 0, G, p.causal);
            const int n = item_tiles(w, x);
            if (n == 0) continue;
            const uint32_t last = load_idx + 2 * (uint32_t)n - 1;  // V_{n-1}
            load_idx += 2 * (uint32_t)n;
            const int r0 = x.kv_len - (w.kt0 + n - 1) * BN;  // first row past kv_len
            if (r0 >= BN) continue;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(FIX_READY), fixes & 1, abort_flag,
                                                           p.status));
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(BAR(KV_FULL + last % C::STAGES),
                                                  (last / C::STAGES) & 1, abort_flag, p.status));
            if (!ok) break;
            ++fixes;
            if constexpr (GROUPED)
                zero_group_rows<C::CHUNKS>(sKV + (last % C::STAGES) * C::TILE_BYTES, r0, lane);
            else
                zero_stage_rows<C::CHUNKS, C::CHUNK_BYTES>(sKV + (last % C::STAGES) * C::TILE_BYTES,
                                                           r0, lane);
            mbar_arrive(BAR(V_FIXED));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax / epilogue
        // One thread per packed row.  The running max is kept in log2 units and O, l keep
        // their scale until the max grows by more than kRescaleThreshold, so most tiles
        // neither touch O in tensor memory nor wait for the previous P.V.  A split item
        // (part >= 0) writes its O / l and lse in fp32 for the merge kernel.
        const int r = threadIdx.x - 128;                       // packed row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t o_addr = tmem_base + lane_base + C::TMEM_O;
        const int Hq = p.num_qo_heads;
        const bool fast_scale = p.scale_log2 > 0.f;
        const float c_eff = fast_scale ? p.scale_log2 : 1.f;
        uint32_t tile_ctr = 0, items_done = 0;
        bool ok = true;
        int rr = -1;
        int it = snake_next(rr, n_items);
        while (ok && it >= 0) {
            const WorkItem w = load_item(p.items, it);
            it = snake_next(rr, n_items);
            const Geo x = geo_of(w, 0, G, p.causal);
            const int row_t = x.t0 + r / G;
            const int row_h = w.g * G + r % G;
            const bool valid = row_t < x.qo_len;
            const size_t out_row = (size_t)(x.q_start + row_t) * Hq + row_h;
            const int n = item_tiles(w, x);
            if (n == 0) {
                // no visible key: zeros (a chunk of a split request without keys for this
                // tile writes nothing; the merge leaves that chunk out)
                if (valid && w.part < 0) {
                    uint4* op = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                         out_row * D);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[out_row] = -INFINITY;
                }
                continue;
            }
            const int klim = p.causal ? min(row_t + x.kv_len - x.qo_len, x.kv_len - 1)
                                      : x.kv_len - 1;
            float m_used = -INFINITY, l = 0.f;
            for (int jr = 0; jr < n; ++jr) {
                const int j = w.kt0 + jr;  // absolute K/V tile (masking)
                const uint32_t ctr = tile_ctr + jr;
                const uint32_t buf = ctr & 1;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(S_FULL + buf), (ctr >> 1) & 1,
                                                               abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_addr = tmem_base + lane_base + (buf ? 128u : 0u);
                uint32_t u[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_addr + cc * 32, u[cc]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_wait_ld_regs(u[cc]);
                float s[BN];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(u[cc][i]);
                if (!fast_scale) {
                    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
                    for (int i = 0; i < BN; i += 2)
                        f2_unpack(f2_mul(f2_pack(s[i], s[i + 1]), c2), s[i], s[i + 1]);
                }
                if (j >= x.n_unmasked) {
                    const int key0 = j * BN;
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (key0 + i > klim) s[i] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx[q] = fmaxf(s[q], s[8 + q]);
#pragma unroll
                for (int i = 16; i < BN; i += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], s[i + q], s[i + 8 + q]);
                const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                       fmaxf(mx[6], mx[7])) * c_eff;
                const bool grow = mt > m_used + kRescaleThreshold;
                const float m_new = grow ? mt : m_used;
                const float alpha = grow ? ex2_approx(m_used - m_new) : 1.f;
                const float neg = m_new == -INFINITY ? 0.f : -m_new;
                const uint64_t c2 = f2_pack(c_eff, c_eff), n2 = f2_pack(neg, neg);
                uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = cc * 64 + 2 * i;
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), c2, n2), t0, t1);
                        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                        if (i & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
                        else acc0 = f2_add(acc0, f2_pack(p0, p1));
                        pk[i] = F8CONV ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + cc * 32, pk);
                }
                float a0, a1, a2, a3;
                f2_unpack(acc0, a0, a1);
                f2_unpack(acc1, a2, a3);
                l = l * alpha + ((a0 + a1) + (a2 + a3));
                if (jr > 0 && __any_sync(0xffffffffu, grow)) {
                    // the previous tile's P.V must be done before O is rescaled
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(PV_DONE), (ctr - 1) & 1,
                                                                   abort_flag, p.status));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
                    for (int oc = 0; oc < D / 32; ++oc) {
                        uint32_t v[32];
                        tmem_ld32(o_addr + oc * 32, v);
                        tmem_wait_ld_regs(v);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float o0, o1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                             al2), o0, o1);
                            v[i] = __float_as_uint(o0);
                            v[i + 1] = __float_as_uint(o1);
                        }
                        tmem_st32(o_addr + oc * 32, v);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR(P_FULL + buf));
                m_used = m_new;
            }
            if (!ok) break;
            tile_ctr += n;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(PV_LAST), items_done & 1,
                                                           abort_flag, p.status));
            ++items_done;
            if (!ok) break;
            tc_fence_after();
            const float inv_l = l > 0.f ? p.v_scale / l : 0.f;
            const float lse_v = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
            if (w.part >= 0) {
                // split-KV partial: O / l in fp32 and the chunk's lse
                const long long slot = (long long)w.part + (long long)row_t * Hq + row_h;
                float4* op = reinterpret_cast<float4*>(p.part_o + slot * D);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
                    tmem_wait_ld_regs(v);
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            op[c * 8 + e] = make_float4(__uint_as_float(v[4 * e]) * inv_l,
                                                        __uint_as_float(v[4 * e + 1]) * inv_l,
                                                        __uint_as_float(v[4 * e + 2]) * inv_l,
                                                        __uint_as_float(v[4 * e + 3]) * inv_l);
                    }
                }
                if (valid) p.part_lse[slot] = lse_v;
            } else {
                uint4* op = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                     out_row * D);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
                    tmem_wait_ld_regs(v);
                    if (valid) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 q;
                            q.x = pack_bf16x2(__uint_as_float(v[v4 * 8 + 0]) * inv_l,
                                              __uint_as_float(v[v4 * 8 + 1]) * inv_l);
                            q.y = pack_bf16x2(__uint_as_float(v[v4 * 8 + 2]) * inv_l,
                                              __uint_as_float(v[v4 * 8 + 3]) * inv_l);
                            q.z = pack_bf16x2(__uint_as_float(v[v4 * 8 + 4]) * inv_l,
                                              __uint_as_float(v[v4 * 8 + 5]) * inv_l);
                            q.w = pack_bf16x2(__uint_as_float(v[v4 * 8 + 6]) * inv_l,
                                              __uint_as_float(v[v4 * 8 + 7]) * inv_l);
                            op[c * 4 + v4] = q;
                        }
                    }
                }
                if (valid && p.lse) p.lse[out_row] = lse_v;
            }
            tc_fence_before();
            mbar_arrive(BAR(O_EMPTY));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------ two-tile kernel (hd128)
// One work item = two consecutive q tiles (A, B) of one (request, kv head).  Both tiles
// share every K/V tile the producer streams in, so K/V shared-memory traffic per flop
// halves, and the tensor core alternates between the two tiles: while warpgroup A runs
// the softmax of its tile, the MMA warp runs B's P.V and Q.K^T, and vice versa.
// TMEM columns: S_A 0..127, S_B 128..255, O_A 256..383, O_B 384..511.
struct PairCfg {
    static constexpr int D = 128;
    static constexpr int CHUNKS = 2;
    static constexpr int CHUNK_BYTES = BM * 128;
    static constexpr int TILE_BYTES = BM * D * 2;
    static constexpr int STAGES = 4;
    static constexpr int NUM_BARS = 17;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES * (2 + STAGES) + 8 * NUM_BARS + 16;
};


// F8CONV: K/V pages converted from an E4M3 cache (V to f16): the output takes p.v_scale,
// P is rounded to f16 and P.V runs on f16 operands; a separate instance, so the bf16 paths
// keep their code unchanged
template <bool PAGED, bool F8CONV>
__global__ void __launch_bounds__(PAIR_THREADS, 1) attention_pair_kernel(const Params p) {
    using C = PairCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);  // tile A at sQ, tile B at sQ + TILE_BYTES
    const uint32_t sKV = sQ + 2 * C::TILE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE_BYTES * (2 + C::STAGES));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    // STEP_FULL[t % 2]: the K/V tiles one MMA step consumes have landed (TMA tx count);
    // A step's stages are free again once its last MMA group has completed: that group's
    // commit is S_FULL of tile B (tile A for items without B) or, on an item's final step,
    // PV_DONE; the producer waits on those, so the MMA warp issues no extra commit.
    // S_FULL[2x + c % 2]: Q.K^T of tile x's c-th K/V tile is in tensor memory.  Two
    // barriers per tile, alternating: the producer waits for step t's completion only
    // after it has issued step t + 1, so with one barrier per tile the completions of
    // steps t and t + 1 could both land before it looks and its parity wait would miss
    // them.  The next completion on the same barrier needs step t + 2's loads, which the
    // producer issues only after that wait.
    // Paged K/V only: slots past kv_len in an item's last V tile hold whatever the cache
    // holds there (or stale data of an earlier tile), and P.V would turn a NaN there into
    // a NaN result even with P = 0.  The producer arrives on FIX_READY once it has issued
    // the loads of such a last step; warp 2 then waits for them, zeroes those V rows and
    // arrives on V_FIXED, which the MMA warp waits for instead of the step's STEP_FULL.
    // P_LO[x]: the first half of tile x's P (keys 0..63) is in tensor memory; P_FULL[x]:
    // all of it.  The MMA warp issues the P.V of each half as soon as that half is there.
    constexpr int Q_FULL = 0, Q_EMPTY = 1, STEP_FULL = 2, S_FULL = 4,
                  P_FULL = S_FULL + 4, PV_DONE = P_FULL + 2, MMA_DRAIN = PV_DONE + 2,
                  FIX_READY = MMA_DRAIN + 1, V_FIXED = FIX_READY + 1, P_LO = V_FIXED + 1;
    static_assert(P_LO + 2 == C::NUM_BARS, "barrier count");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(BAR(Q_FULL), 1);
        mbar_init(BAR(Q_EMPTY), 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(STEP_FULL + x), 1);
            mbar_init(BAR(S_FULL + 2 * x), 1);
            mbar_init(BAR(S_FULL + 2 * x + 1), 1);
            mbar_init(BAR(P_FULL + x), 128);
            mbar_init(BAR(P_LO + x), 128);
            mbar_init(BAR(PV_DONE + x), 1);
        }
        mbar_init(BAR(MMA_DRAIN), 1);
        mbar_init(BAR(FIX_READY), 1);
        mbar_init(BAR(V_FIXED), 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the prologue above overlapped the plan kernel; its outputs are read from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = __ldcg(&p.hdr->n_items);  // written by the plan
    const int G = p.group;
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // An item of n K/V tiles is n + 1 MMA steps: step t consumes V_{t-1} and K_t.  The
        // loads of step t go out once step t - 2 is done, which frees both their stages.
        // Ragged K/V: lane 0 alone.  Paged K/V: the whole warp, lane l loading page l of
        // each K/V tile (its id read one step ahead); lane 0 arms the barriers.
        if (PAGED || lane == 0) {
            auto wait = [&](uint32_t bar, uint32_t par) -> bool {
                if constexpr (PAGED)
                    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, par, abort_flag, p.status));
                else
                    return mbar_wait_bounded(bar, par, abort_flag, p.status);
            };
            tensormap_acquire(p.tm_q);
            tensormap_acquire(p.tm_k);
            tensormap_acquire(p.tm_v);
            const int ps = p.page_size;
            const int ppt = PAGED ? BN / ps : 0;
            uint32_t load_idx = 0, q_count = 0, step = 0;
            uint32_t ctr[2] = {0, 0}, items_x[2] = {0, 0};
            uint32_t done_bar[2] = {0, 0}, done_par[2] = {0, 0};  // completion of steps t, t-1
            bool ok = true;
            int rr = -1;
            int it = snake_next(rr, n_items);
            while (ok && it >= 0) {
                const WorkItem w = load_item(p.items, it);
                it = snake_next(rr, n_items);
                const Geo a = geo_of(w, 0, G, p.causal);
                const Geo bq = geo_of(w, 1, G, p.causal);
                const int nA = item_tiles(w, a);
                const int nB = bq.t0 < bq.qo_len ? item_tiles(w, bq) : 0;
                const int nmax = max(nA, nB);
                if (nmax == 0) continue;
                const int lx = nB > 0 ? 1 : 0;  // tile whose MMAs close every step
                const int kt0 = w.kt0;          // first K/V tile of the item
                ok = wait(BAR(Q_EMPTY), (q_count & 1) ^ 1);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(BAR(Q_FULL), C::TILE_BYTES * (nB > 0 ? 2 : 1));
#pragma unroll
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tma_load_3d(sQ + c * C::CHUNK_BYTES, p.tm_q, BAR(Q_FULL), c * 64, w.g * G,
                                    a.q_start + a.t0);
                    if (nB > 0) {
#pragma unroll
                        for (int c = 0; c < C::CHUNKS; ++c)
                            tma_load_3d(sQ + C::TILE_BYTES + c * C::CHUNK_BYTES, p.tm_q,
                                        BAR(Q_FULL), c * 64, w.g * G, bq.q_start + bq.t0);
                    }
                }
                ++q_count;
                const uint32_t L0 = load_idx;
                const int* pt_row = PAGED ? p.page_table + (size_t)w.b * p.page_table_stride : nullptr;
                const int npg = PAGED ? (a.kv_len + ps - 1) / ps : 0;
                // paged: this lane's page of K_t (read a step ahead) and of K_{t-1} (= V_{t-1})
                int kid = PAGED ? lane_page_id(pt_row, kt0, ppt, npg, lane) : -1;
                int vid = -1;
                bool v_ok = false;
                for (int t = 0; t <= nmax; ++t, ++step) {
                    if (step >= 2) {
                        ok = wait(done_bar[step & 1], done_par[step & 1]);
                        if (!ok) break;
                    }
                    if (t < nmax) {
                        const uint32_t c = ctr[lx] + t;
                        done_bar[step & 1] = BAR(S_FULL + 2 * lx + (c & 1));
                        done_par[step & 1] = (c >> 1) & 1;
                    } else {
                        done_bar[step & 1] = BAR(PV_DONE + lx);
                        done_par[step & 1] = items_x[lx] & 1;
                    }
                    const uint32_t bar = BAR(STEP_FULL + (step & 1));
                    const uint32_t vst = (L0 + 2 * (t - 1) + 1) % C::STAGES;
                    const uint32_t kst = (L0 + 2 * t) % C::STAGES;
                    if constexpr (PAGED) {
                        const bool k_ok = t < nmax && lane_page_ok(kid, kt0 + t, ppt, npg,
                                                                   p.num_pages, lane, p.status);
                        issue_page_boxes<C::CHUNKS, C::CHUNK_BYTES>(
                            bar, ps, w.g, lane, t >= 1 && v_ok, sKV + vst * C::TILE_BYTES, p.tm_v,
                            vid, k_ok, sKV + kst * C::TILE_BYTES, p.tm_k, kid);
                        if (lane == 0 && t == nmax && (kt0 + nmax) * BN > a.kv_len)
                            mbar_arrive(BAR(FIX_READY));
                        vid = kid;
                        v_ok = k_ok;
                        if (t + 1 < nmax) kid = lane_page_id(pt_row, kt0 + t + 1, ppt, npg, lane);
                    } else {
                        mbar_arrive_expect_tx(bar, C::TILE_BYTES * ((t >= 1) + (t < nmax)));
                        if (t >= 1) {  // V_{t-1}
#pragma unroll
                            for (int c = 0; c < C::CHUNKS; ++c)
                                tma_load_2d(sKV + vst * C::TILE_BYTES + c * C::CHUNK_BYTES, p.tm_v,
                                            bar, w.g * D + c * 64, a.kv_start + (kt0 + t - 1) * BN);
                        }
                        if (t < nmax) {  // K_t
#pragma unroll
                            for (int c = 0; c < C::CHUNKS; ++c)
                                tma_load_2d(sKV + kst * C::TILE_BYTES + c * C::CHUNK_BYTES, p.tm_k,
                                            bar, w.g * D + c * 64, a.kv_start + (kt0 + t) * BN);
                        }
                    }
                }
                load_idx = L0 + 2 * nmax;
                ctr[0] += nA;
                ctr[1] += nB;
                if (nA > 0) ++items_x[0];
                if (nB > 0) ++items_x[1];
            }
            if (!ok && lane == 0) {
                // let every copy already issued land before the CTA exits
                for (uint32_t s = step > 2 ? step - 2 : 0; s < step; ++s)
                    mbar_wait_bounded(BAR(STEP_FULL + (s & 1)), (s >> 1) & 1, nullptr, p.status);
                if (q_count > 0)
                    mbar_wait_bounded(BAR(Q_FULL), (q_count - 1) & 1, nullptr, p.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Step t of an item: P.V of A's tile t-1, Q.K^T of A's tile t, then the same for B.
        // tcgen05.mma issue paces the tensor core, so this thread keeps its own waits and
        // commits per step to a minimum: one wait for the step's K/V, two per P tile (one
        // per half), and commits for S_A, S_B and the step (PV_DONE only after an item's
        // last P.V).
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t IDESC_PV =
                F8CONV ? idesc_f16_f32(BM, D, true) : idesc_bf16_f32(BM, D, true);
            const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
            uint32_t load_idx = 0, q_count = 0, step = 0, fixes = 0;
            uint32_t ctr[2] = {0, 0}, items_x[2] = {0, 0};
            bool ok = true;
            int rr = -1;
            int it = snake_next(rr, n_items);
            while (ok && it >= 0) {
                const WorkItem w = load_item(p.items, it);
                it = snake_next(rr, n_items);
                const Geo a = geo_of(w, 0, G, p.causal);
                const Geo bq = geo_of(w, 1, G, p.causal);
                const int nx[2] = {item_tiles(w, a), bq.t0 < bq.qo_len ? item_tiles(w, bq) : 0};
                const int nmax = max(nx[0], nx[1]);
                if (nmax == 0) continue;
                ok = mbar_wait_bounded(BAR(Q_FULL), q_count & 1, abort_flag, p.status);
                ++q_count;
                if (!ok) break;
                const uint32_t L0 = load_idx;
                const bool fix = PAGED && (w.kt0 + nmax) * BN > a.kv_len;
                for (int t = 0; t <= nmax; ++t, ++step) {
                    if (fix && t == nmax) {  // the last V tile, its tail rows zeroed
                        ok = mbar_wait_bounded(BAR(V_FIXED), fixes & 1, abort_flag, p.status);
                        ++fixes;
                    } else {
                        ok = mbar_wait_bounded(BAR(STEP_FULL + (step & 1)), (step >> 1) & 1,
                                               abort_flag, p.status);
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vst = (L0 + 2 * (t - 1) + 1) % C::STAGES;
                    const uint32_t kst = (L0 + 2 * t) % C::STAGES;
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (t >= 1 && t - 1 < nx[x]) {
                            const int jj = t - 1;
                            // P_LO of an item's first tile also says that the previous
                            // item's O has been read out, so this P.V may overwrite it
                            // descriptor of a 16-key slice = base + byte offset / 16
                            const uint64_t vdesc =
                                sdesc_sw128(sKV + vst * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
                            // P in two halves: keys 0..63 (P_LO), then 64..127 (P_FULL)
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                ok = mbar_wait_bounded(BAR((hf ? P_FULL : P_LO) + x),
                                                       (ctr[x] + jj) & 1, abort_flag, p.status);
                                if (!ok) break;
                                tc_fence_after();
#pragma unroll
                                for (int k = hf * BN / 32; k < (hf + 1) * BN / 32; ++k)
                                    mma_ts(tmem_base + 256u + 128u * x, tmem_base + 128u * x + k * 8,
                                           vdesc + (uint64_t)(k * 2048 / 16), IDESC_PV,
                                           (jj > 0 || k > 0) ? 1u : 0u);
                            }
                            if (!ok) break;
                            if (jj == nx[x] - 1) mma_commit(BAR(PV_DONE + x));
                        }
                        if (t < nx[x]) {
                            const uint64_t kdesc = sdesc_sw128(sKV + kst * C::TILE_BYTES, 16, 1024);
                            const uint64_t qdesc = qdesc0 + (uint64_t)(x * C::TILE_BYTES / 16);
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint64_t off = ((k >> 2) * C::CHUNK_BYTES + (k & 3) * 32) / 16;
                                mma_ss(tmem_base + 128u * x, qdesc + off, kdesc + off, IDESC_QK,
                                       k > 0 ? 1u : 0u);
                            }
                            mma_commit(BAR(S_FULL + 2 * x + ((ctr[x] + t) & 1)));
                        }
                    }
                    if (!ok) break;
                    if (t == nmax - 1) mma_commit(BAR(Q_EMPTY));
                }
                if (!ok) break;
                load_idx = L0 + 2 * nmax;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    ctr[x] += nx[x];
                    if (nx[x] > 0) ++items_x[x];
                }
            }
            // every MMA issued has completed before tensor memory is released
            mma_commit(BAR(MMA_DRAIN));
            mbar_wait_bounded(BAR(MMA_DRAIN), 0, nullptr, p.status);
        }
    } else if (PAGED && warp == 2) {
        // ------------------------------------------------------------ V tail fixer
        uint32_t step = 0, load_idx = 0, fixes = 0;
        bool ok = true;
        int rr = -1;
        int it = snake_next(rr, n_items);
        while (ok && it >= 0) {
            const WorkItem w = load_item(p.items, it);
            it = snake_next(rr, n_items);
            const Geo a = geo_of(w, 0, G, p.causal);
            const Geo bq = geo_of(w, 1, G, p.causal);
            const int nmax = max(item_tiles(w, a), bq.t0 < bq.qo_len ? item_tiles(w, bq) : 0);
            if (nmax == 0) continue;
            const uint32_t L0 = load_idx;
            const uint32_t fin = step + (uint32_t)nmax;  // the item's last step: V_{nmax-1}
            step += (uint32_t)nmax + 1;
            load_idx = L0 + 2 * (uint32_t)nmax;
            const int last = w.kt0 + nmax - 1;           // absolute index of that V tile
            if ((last + 1) * BN <= a.kv_len) continue;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(FIX_READY), fixes & 1, abort_flag,
                                                           p.status));
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(BAR(STEP_FULL + (fin & 1)), (fin >> 1) & 1,
                                                  abort_flag, p.status));
            if (!ok) break;
            ++fixes;
            const uint32_t st = (L0 + 2 * (uint32_t)(nmax - 1) + 1) % C::STAGES;
            zero_stage_rows<C::CHUNKS, C::CHUNK_BYTES>(sKV + st * C::TILE_BYTES,
                                                       a.kv_len - last * BN, lane);
            mbar_arrive(BAR(V_FIXED));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax / epilogue
        // The epilogue of an item (O / l -> bf16 rows, lse) runs inside the next item's
        // first tile: once that tile's P is in tensor memory, the warpgroup reads the
        // previous O, releases O and P together, and then stores, so the stores overlap the
        // tensor core's next P.V instead of delaying it.
        const int X = warp >= 8 ? 1 : 0;
        const int r = threadIdx.x - 128 - 128 * X;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t s_addr = tmem_base + lane_base + 128u * X;
        const uint32_t o_addr = tmem_base + lane_base + 256u + 128u * X;
        const int Hq = p.num_qo_heads;
        const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;
        const bool fast_scale = p.scale_log2 > 0.f;
        const float c_eff = fast_scale ? p.scale_log2 : 1.f;
        uint32_t ctr = 0, items_done = 0;
        // the item whose epilogue is pending (pend_slot >= 0: a partial-result row)
        bool pend = false, pend_valid = false;
        float pend_l = 0.f, pend_m = 0.f;
        size_t pend_row = 0;
        long long pend_slot = -1;
        // Wait for the pending item's last P.V and read its O row out of tensor memory.
        auto read_pending = [&](uint32_t (&u)[4][32]) -> bool {
            const bool okw = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(PV_DONE + X),
                                                                        items_done & 1,
                                                                        abort_flag, p.status));
            ++items_done;
            if (!okw) return false;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(o_addr + cc * 32, u[cc]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_wait_ld_regs(u[cc]);
            return true;
        };
        auto store_pending = [&](const uint32_t (&u)[4][32]) {
            if (!pend_valid) return;
            const float inv_l = pend_l > 0.f ? (F8CONV ? p.v_scale : 1.f) / pend_l : 0.f;
            if (pend_slot >= 0) {  // split-KV partial: O / l in fp32 and the chunk's lse
                float4* op = reinterpret_cast<float4*>(p.part_o + pend_slot * D);
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        op[cc * 8 + e] = make_float4(__uint_as_float(u[cc][4 * e]) * inv_l,
                                                     __uint_as_float(u[cc][4 * e + 1]) * inv_l,
                                                     __uint_as_float(u[cc][4 * e + 2]) * inv_l,
                                                     __uint_as_float(u[cc][4 * e + 3]) * inv_l);
                p.part_lse[pend_slot] =
                    pend_l > 0.f ? (pend_m + log2f(pend_l)) * 0.69314718055994531f : -INFINITY;
                return;
            }
            uint4* op = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + pend_row * D);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(u[cc][2 * e]) * inv_l,
                                        __uint_as_float(u[cc][2 * e + 1]) * inv_l);
                if (o32) {  // 32-byte stores: whole sectors, half the store instructions
#pragma unroll
                    for (int h = 0; h < 2; ++h) st_global_v8(op + cc * 4 + h * 2, pk + 8 * h);
                } else {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        op[cc * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                                     pk[4 * v4 + 3]);
                }
            }
            if (p.lse)
                p.lse[pend_row] =
                    pend_l > 0.f ? (pend_m + log2f(pend_l)) * 0.69314718055994531f : -INFINITY;
        };
        bool ok = true;
        int rr = -1;
        int it = snake_next(rr, n_items);
        while (ok && it >= 0) {
            const WorkItem w = load_item(p.items, it);
            it = snake_next(rr, n_items);
            const Geo x = geo_of(w, X, G, p.causal);
            if (x.t0 >= x.qo_len) continue;  // this item has no tile B
            const int row_t = x.t0 + r / G;
            const int row_h = w.g * G + r % G;
            const bool valid = row_t < x.qo_len;
            const size_t out_row = (size_t)(x.q_start + row_t) * Hq + row_h;
            const int nt = item_tiles(w, x);
            if (nt == 0) {
                // no visible key: zeros (a chunk of a split request without keys for this
                // tile writes nothing; the merge leaves that chunk out)
                if (valid && w.part < 0) {
                    uint4* op = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                         out_row * D);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) op[c] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[out_row] = -INFINITY;
                }
                continue;
            }
            const int klim = p.causal ? min(row_t + x.kv_len - x.qo_len, x.kv_len - 1)
                                      : x.kv_len - 1;
            float m_used = -INFINITY, l = 0.f;
            for (int jr = 0; jr < nt; ++jr) {
                const int j = w.kt0 + jr;  // absolute K/V tile (masking); jr: within the item
                const uint32_t c = ctr + jr;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(S_FULL + 2 * X + (c & 1)),
                                                               (c >> 1) & 1, abort_flag,
                                                               p.status));
                if (!ok) break;
                tc_fence_after();
                // S row: four 32-column TMEM loads in flight, one wait
                uint32_t u[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_addr + cc * 32, u[cc]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_wait_ld_regs(u[cc]);
                float s[BN];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(u[cc][i]);
                if (!fast_scale) {
                    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
                    for (int i = 0; i < BN; i += 2)
                        f2_unpack(f2_mul(f2_pack(s[i], s[i + 1]), c2), s[i], s[i + 1]);
                }
                if (j >= x.n_unmasked) {
                    const int key0 = j * BN;
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (key0 + i > klim) s[i] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[k], s[8 + k]);
#pragma unroll
                for (int i = 16; i < BN; i += 16)
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[i + k], s[i + 8 + k]);
                const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                       fmaxf(mx[6], mx[7])) * c_eff;
                const bool grow = mt > m_used + kRescaleThreshold;
                const float m_new = grow ? mt : m_used;
                const float alpha = grow ? ex2_approx(m_used - m_new) : 1.f;
                const float neg = m_new == -INFINITY ? 0.f : -m_new;
                const uint64_t c2 = f2_pack(c_eff, c_eff), n2 = f2_pack(neg, neg);
                uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
                // P leaves in two halves (P_LO: keys 0..63) so that the tensor core starts
                // this tile's P.V while the second half is computed.  The first tile of an
                // item with an epilogue pending releases both halves only after the
                // previous O has been read out.
                const bool early = jr > 0 || !pend;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = cc * 64 + 2 * i;
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), c2, n2), t0, t1);
                        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                        if (i & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
                        else acc0 = f2_add(acc0, f2_pack(p0, p1));
                        pk[i] = F8CONV ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + cc * 32, pk);
                    if (cc == 0 && early) {
                        // O may be rescaled now: S_FULL of this tile was committed after the
                        // previous P.V by the same issuing thread, so that P.V has completed
                        if (jr > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
                            for (int oc = 0; oc < D / 32; ++oc) {
                                uint32_t v[32];
                                tmem_ld32(o_addr + oc * 32, v);
                                tmem_wait_ld_regs(v);
                                const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
                                for (int i = 0; i < 32; i += 2) {
                                    float o0, o1;
                                    f2_unpack(f2_mul(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), al2), o0, o1);
                                    v[i] = __float_as_uint(o0);
                                    v[i + 1] = __float_as_uint(o1);
                                }
                                tmem_st32(o_addr + oc * 32, v);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(BAR(P_LO + X));
                    }
                }
                float a0, a1, a2, a3;
                f2_unpack(acc0, a0, a1);
                f2_unpack(acc1, a2, a3);
                l = l * alpha + ((a0 + a1) + (a2 + a3));
                if (early) {
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(BAR(P_FULL + X));
                } else {
                    // first tile of an item with an epilogue pending: read the previous O
                    // (its last P.V is done), release O and this tile's P, then store
                    ok = read_pending(u);
                    if (!ok) break;
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(BAR(P_LO + X));
                    mbar_arrive(BAR(P_FULL + X));
                    store_pending(u);
                }
                m_used = m_new;
            }
            if (!ok) break;
            ctr += nt;
            pend = true;
            pend_valid = valid;
            pend_l = l;
            pend_m = m_used;
            pend_row = out_row;
            pend_slot = w.part >= 0 ? (long long)w.part + (long long)row_t * Hq + row_h : -1;
        }
        if (ok && pend) {
            uint32_t u[4][32];
            if (read_pending(u)) store_pending(u);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------ split-KV merge
// One warp per (token, query head) row of a split request: the chunks that hold keys
// visible to the row are combined with weights exp(lse_c - max lse) (FlashInfer
// documentation, flashinfer.cascade "Merge Attention States").  Rows without a visible key
// get zeros and lse = -inf.  Lane l combines columns 4l .. 4l + 3 of each 128-column half.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const Params p) {
    constexpr int NV = D / 128;  // float4s per lane
    // launched as a dependent of the attention kernel: its partial results are read from here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int rows = p.hdr->merge_rows;
    const int Hq = p.num_qo_heads;
    const int lane = threadIdx.x & 31;
    for (long long m = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); m < rows;
         m += (long long)gridDim.x * 8) {
        const int b = find_segment(p.merge_off, p.batch, (int)m);
        const int local = (int)m - __ldg(p.merge_off + b);
        const int t = local / Hq, h = local % Hq;
        const int q0 = __ldg(p.q_indptr + b);
        const int qo = __ldg(p.q_indptr + b + 1) - q0;
        const int kv = __ldg(p.kvl + b);
        const int nc = __ldg(p.nch + b);
        const int nkeys = p.causal ? max(0, min(kv, t + kv - qo + 1)) : kv;
        const int nvis = min(nc, (nkeys + p.split_tiles * BN - 1) / (p.split_tiles * BN));
        const long long base = __ldg(p.part_off + b);
        auto slot = [&](int c) { return base + ((long long)c * qo + t) * Hq + h; };
        float mx = -INFINITY;
        for (int c = lane; c < nvis; c += 32) mx = fmaxf(mx, p.part_lse[slot(c)]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float4 acc[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (mx != -INFINITY) {
            // chunks in index order, the loads of MU chunks issued before their arithmetic
            constexpr int MU = 4;
            auto add = [&](float l, const float4 (&v)[NV]) {
                const float wgt = __expf(l - mx);
                wsum += wgt;
#pragma unroll
                for (int e = 0; e < NV; ++e) {
                    acc[e].x = fmaf(wgt, v[e].x, acc[e].x);
                    acc[e].y = fmaf(wgt, v[e].y, acc[e].y);
                    acc[e].z = fmaf(wgt, v[e].z, acc[e].z);
                    acc[e].w = fmaf(wgt, v[e].w, acc[e].w);
                }
            };
            auto row = [&](int c, float4 (&v)[NV]) {
                const float4* r = reinterpret_cast<const float4*>(p.part_o + slot(c) * D);
#pragma unroll
                for (int e = 0; e < NV; ++e) v[e] = r[e * 32 + lane];
            };
            int c = 0;
            for (; c + MU <= nvis; c += MU) {
                float l[MU];
                float4 v[MU][NV];
#pragma unroll
                for (int u = 0; u < MU; ++u) {
                    l[u] = p.part_lse[slot(c + u)];
                    row(c + u, v[u]);
                }
#pragma unroll
                for (int u = 0; u < MU; ++u) add(l[u], v[u]);
            }
            for (; c < nvis; ++c) {
                float4 v[NV];
                row(c, v);
                add(p.part_lse[slot(c)], v);
            }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)(q0 + t) * Hq + h) * D;
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            uint2 u;
            u.x = pack_bf16x2(acc[e].x * inv, acc[e].y * inv);
            u.y = pack_bf16x2(acc[e].z * inv, acc[e].w * inv);
            *reinterpret_cast<uint2*>(op + e * 128 + lane * 4) = u;
        }
        if (lane == 0 && p.lse)
            p.lse[(size_t)(q0 + t) * Hq + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
    }
}

// ------------------------------------------------------------------ host launchers
// The attention and merge kernels are launched with launch_dependent (ptx.cuh): they may
// start while the plan still runs and execute griddepcontrol.wait before using its output.

template <int D, bool PAGED, bool GROUPED, bool F8CONV>
static cudaError_t launch_attention_t(const Params& p, int grid, cudaStream_t stream) {
    static std::atomic<bool> configured[64];  // per device, set once (repeats are harmless)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<D, PAGED, GROUPED, F8CONV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<D>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    return launch_dependent(attention_kernel<D, PAGED, GROUPED, F8CONV>, grid, THREADS,
                            Cfg<D>::SMEM_BYTES, stream, p);
}

// grouped: paged K/V through 5-D tensor maps filling the grouped stage layout; p.f8conv:
// pages converted from an E4M3 cache
template <int D, bool PAGED>
cudaError_t launch_attention(const Params& p, int grid, bool grouped, cudaStream_t stream) {
    if constexpr (PAGED) {
        if (p.f8conv)
            return grouped ? launch_attention_t<D, true, true, true>(p, grid, stream)
                           : launch_attention_t<D, true, false, true>(p, grid, stream);
        if (grouped) return launch_attention_t<D, true, true, false>(p, grid, stream);
    }
    return launch_attention_t<D, PAGED, false, false>(p, grid, stream);
}

template <bool PAGED, bool F8CONV>
static cudaError_t launch_pair_t(const Params& p, int grid, cudaStream_t stream) {
    static std::atomic<bool> configured[64];  // per device, set once (repeats are harmless)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(attention_pair_kernel<PAGED, F8CONV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             PairCfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    return launch_dependent(attention_pair_kernel<PAGED, F8CONV>, grid, PAIR_THREADS,
                            PairCfg::SMEM_BYTES, stream, p);
}

template <bool PAGED>
cudaError_t launch_attention_pair(const Params& p, int grid, cudaStream_t stream) {
    if constexpr (PAGED) {
        if (p.f8conv) return launch_pair_t<true, true>(p, grid, stream);
    }
    return launch_pair_t<PAGED, false>(p, grid, stream);
}

cudaError_t launch_merge(const Params& p, int head_dim, int num_sms, cudaStream_t stream) {
    return head_dim == 256 ? launch_dependent(merge_kernel<256>, num_sms * 2, 256, 0, stream, p)
                           : launch_dependent(merge_kernel<128>, num_sms * 2, 256, 0, stream, p);
}

cudaError_t launch_plan(const PlanParams& pp, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, cudaStream_t stream) {
    constexpr int kDyn = PLAN_STAGE_UNITS * (int)sizeof(WorkItem);
    static std::atomic<bool> attr_set[64];  // per device, set once (repeats are harmless)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    plan_kernel<<<1, PLAN_THREADS, kDyn, stream>>>(pp, tq, tk, tv);
    return cudaGetLastError();
}

template cudaError_t launch_attention<256, false>(const Params&, int, bool, cudaStream_t);
template cudaError_t launch_attention<256, true>(const Params&, int, bool, cudaStream_t);
template cudaError_t launch_attention_pair<false>(const Params&, int, cudaStream_t);
template cudaError_t launch_attention_pair<true>(const Params&, int, cudaStream_t);

}  // namespace prefill
}  // namespace pgqa
