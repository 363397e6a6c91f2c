// decode_mma.cu -- paged GQA decode over an FP8 E4M3 KV cache on the tensor cores.
//
// What it computes is the decode of decode.cu (one query row per request; split-KV over
// request-local chunks; partial results merged by log-sum-exp weights) with K/V stored as
// OCP E4M3 bytes and one scale per tensor:
//   o[b,h] = v_scale * softmax_j(sm_scale * k_scale * q[b,h] . k8[j, h/G]) v8[j, h/G]
// and the same for a few query rows per request (a paged prefill of at most 16 / G rows per
// request, as in multi-token decode): row i of a request with qo rows and kv keys sees the
// keys j <= i + kv - qo when causal, all kv keys otherwise.
// Sources: FlashInfer documentation, flashinfer_benchmark.py "Attention Flags"
// (--kv_dtype fp8_e4m3; --causal for the prefill routines); vllm-rlt pull request "feat: add
// FlashInfer attention backend for SM120 decode" (paged decode over a block table, padding
// never visible); FlashInfer documentation, flashinfer.cascade "Merge Attention States"
// (the chunk merge).
//
// Why the E4M3 bytes go to the tensor core as they are: the decode streams each K/V byte
// once, so the kernel is bound by how many bytes each SM keeps in flight.  A stage of the
// TMA ring that has to be converted (to f16, for kind::f16) is held until the conversion
// ends, and with in-order consumption every slow conversion delays the stages behind it.
// Here the MMAs (kind::f8f6f4) read the raw stages: Q . K^T takes the K tile straight from
// the ring, P . V the V tile as an MN-major operand, and a stage is released by the
// commit of its MMAs.  The other operand of each product, Q and P, is given as a pair of
// E4M3 matrices hi + lo (hi = E4M3(x), lo = E4M3(x - hi)) whose products are summed in
// fp32 (in one accumulator, or in two accumulator columns added afterwards): for Q (bf16,
// scaled by a power of two into [2^7, 2^8)) the pair is exact down to 2^-2, for P (scaled
// by 2^8) it keeps about 8 significant bits, as the bf16 prefill's P does.
//
// Design (one persistent CTA per SM, 384 threads; work item = one (chunk, kv head) of up
// to 8 tiles of 128 keys; the items of a CTA run as a software pipeline in which step s
// handles the K tiles of item s and the V tiles of item s - 1):
//  * warps 0, 2 and 3, producers: stream 128-key tiles of E4M3 bytes in step order through
//    a TMA ring of 12 stages (11 with several query rows), each taking every third tile;
//    lane u < 8 loads the 16-key unit u of a tile (a 16-token page, or a slice of a
//    larger page) as one 2 KB box, 128-byte swizzled: 128 rows (keys) of 128 bytes
//    (dims).  Page ids are read one item ahead.
//  * warp 1, lane 0: MMA issuer (swap-AB, keys as M = 128, query columns padded to N =
//    16; with several query rows per request, column n is row n / G, head n % G):
//      S^T_t  = K_t . (Qhi + Qlo)^T     A = raw K tile (K-major), B = Q parts (K-major)
//      O^T   += V_t^T . (Phi + Plo)^T   A = raw V tile (MN-major), B = P^T parts (MN-major)
//    Every S^T tile of an item stays in tensor memory (two item regions of 8 x 16
//    columns), so the softmax sees the whole item at once; O^T takes 16 (or 32) more.
//    Keys past the chunk and units whose page was not loaded must not reach P . V as
//    whatever bytes the stage held (0 * NaN is NaN): before the MMAs of such a V tile this
//    thread zeroes those rows (the last tile of a request: a few per CTA).
//  * warps 8-11, Q: per item, thread d loads dim d of the item's query rows, finds the
//    power of two 2^e that puts max|q| into [2^7, 2^8), writes 2^e q as E4M3 hi/lo
//    operands, records which 16-key units of the item have a valid page and publishes
//    the item's geometry beside them, so the MMA thread and the softmax never walk the
//    request list; they also write the rows of requests without keys.
//  * warps 4-7, softmax: thread r owns key r of every tile (TMEM lane r).  Per item: one
//    pass over all its S^T tiles gives the exact max per column (a transposing warp
//    butterfly and one exchange among the four warps), so no running rescale is needed;
//    then each tile's P^T = 2^8 exp2(s - max) goes to shared memory as E4M3 hi/lo bytes,
//    one row per key that its thread writes with one or two 16-byte stores (a buffer per
//    tile of the item), while the column sums accumulate; at the item's end thread r
//    holds row r of O^T: divided by l, scaled by v_scale, it becomes the bf16 output
//    (single-chunk request) or the fp32 partial and its lse.
//  While the softmax works on item s - 1, the tensor core is already on the K tiles of
//  item s.
#include <atomic>
#include <climits>

#include "ptx.cuh"

namespace pgqa {
namespace decode {
namespace mmad {

constexpr int D = HEAD_DIM;                 // 128
constexpr int TK = 128;                     // keys per tile = the MMA's M
constexpr int NH = 16;                      // query columns, padded = the MMA's N
constexpr int UNITS = TK / PAGE;            // 16-key units per tile (8)
constexpr int MAX_TILES = 8;                // tiles per item (chunks of at most 1024 keys)
constexpr int MAX_TILES_ROWS = CHUNK_E4M3_ROWS / TK;  // ... with several query rows (896 keys)
static_assert(MAX_TILES_ROWS * TK == CHUNK_E4M3_ROWS, "whole tiles");
constexpr int RAW_BYTES = TK * D;           // 16 KB of E4M3 per K or V tile
constexpr int OP_BYTES = NH * 128;          // one E4M3 operand: 16 rows x 128 bytes
constexpr int QP_BYTES = 2 * OP_BYTES;      // its hi and lo parts
constexpr int PRODUCERS = 3;                // TMA producer warps (0, 2 and 3)
constexpr int W_SMX = 4;                    // softmax warps 4-7
constexpr int W_Q = 8;                      // Q warps 8-11
constexpr int THREADS = 12 * 32;
constexpr float P_LOG2_SCALE = 8.f;         // P^T holds 2^8 P
// tensor memory: S^T regions of two items and O^T.  One query row (packed): tiles of 16
// columns, regions of 8 tiles at 0 and 128, O^T at 256 (16 columns).  Several rows: tiles
// of 32 columns (the hi and lo parts of Q side by side), regions of 7 tiles at 0 and 224,
// O^T at 448 (32 columns, the hi and lo parts of P).
constexpr int TMEM_COLS = 512;

// Shared memory.  Every tile of an item has its own P^T buffer, and the softmax writes an
// item's P^T only after the previous item's last P . V has completed (its epilogue waits
// for that), so no buffer needs a release of its own.  Packed (one query row): 8 buffers
// of 2 KB beside a 12-stage raw ring, an item's tiles published at once; several query
// rows: 7 buffers of 4 KB (items of at most 896 keys) beside 11 raw stages, each tile
// published as it is written.
template <bool PACK>
struct Layout {
    static constexpr int RAW_STAGES = PACK ? 12 : 11;
    static constexpr int NPB = PACK ? MAX_TILES : MAX_TILES_ROWS;   // P^T buffers
    static constexpr uint32_t P_STRIDE = PACK ? (uint32_t)OP_BYTES : (uint32_t)QP_BYTES;
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_Q = OFF_RAW + RAW_STAGES * RAW_BYTES;  // two buffers (hi, lo)
    static constexpr int OFF_P = OFF_Q + 2 * QP_BYTES;              // the P^T buffers
    static constexpr int OFF_RED = OFF_P + NPB * (int)P_STRIDE;     // exchange areas (1 KB)
    // loaded-unit bits per raw stage (<= 16 words), the q exponents (2 words at +64) and
    // the per-item unit masks (2 x 64 bits at +72)
    static constexpr int OFF_MASK = OFF_RED + 1024;
    static constexpr int OFF_ITEM = OFF_MASK + 96;  // the items in the two Q buffers
    static constexpr int OFF_BAR = OFF_ITEM + 128;
    // barrier indices; P_FULL: by item parity (packed) or by buffer
    static constexpr int RAW_FULL = 0, RAW_EMPTY = RAW_FULL + RAW_STAGES,
                         Q_FULL = RAW_EMPTY + RAW_STAGES, Q_EMPTY = Q_FULL + 2,
                         S_FULL = Q_EMPTY + 2, S_EMPTY = S_FULL + 2, P_FULL = S_EMPTY + 2,
                         N_PFULL = PACK ? 2 : NPB, PV_LAST = P_FULL + N_PFULL,
                         O_EMPTY = PV_LAST + 1, MMA_DRAIN = O_EMPTY + 1, XCH_Q = MMA_DRAIN + 1,
                         XCH_SMX = XCH_Q + 1, NUM_BARS = XCH_SMX + 1;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(RAW_STAGES <= 16, "unit-mask words");
    static_assert(OFF_P % 1024 == 0 && P_STRIDE % 1024 == 0, "operand alignment");
};

// Byte (row, col) of a 128-byte-swizzled K-major E4M3 operand (rows of 128 bytes, 16-byte
// units XORed with row % 8, 8-row groups 1 KB apart).
__device__ __forceinline__ uint32_t sw128_byte(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 4) ^ (row & 7))) << 4) + (col & 15));
}

// Geometry of work item `item`: request b, kv head g, chunk f (of the request's nch),
// keys [tok0, tok1) of the request's kv; its query rows q0 .. q0 + qo - 1.  An item with
// no query rows has no tiles.
struct Item {
    int b, g, f, nch, tok0, tok1, ntiles, kv, q0, qo;
};
// A role's position in the request list: request b, whose first chunk is c0.  Every role
// visits its items in increasing order, so the request of the next item is found by
// walking forward from here.
struct Cursor {
    int b = 0, c0 = 0;
};
__device__ __forceinline__ Item item_of(const Params& p, long long item, Cursor& cur) {
    Item it;
    const int Hk = p.num_kv_heads;
    it.f = (int)(item / Hk);
    it.g = (int)(item % Hk);
    // the request whose chunks contain f: the next four chunk offsets are loaded at once
    // (one round trip, where a binary search over the batch takes one per step); only a
    // longer jump falls back to the search.  Every request has at least one chunk.
    int b = cur.b, c0 = cur.c0;
    int nb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        nb[k] = b + 1 + k < p.batch ? __ldg(p.chunk_off + b + 1 + k) : INT_MAX;
    int adv = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) adv += nb[k] <= it.f ? 1 : 0;
    int c1;
    if (adv < 4) {
        if (adv > 0) c0 = nb[adv - 1];
        b += adv;
        c1 = nb[adv];
    } else {
        int lo = b + 4, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.chunk_off + mid) <= it.f) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
        c0 = __ldg(p.chunk_off + b);
        c1 = __ldg(p.chunk_off + b + 1);
    }
    if (b + 1 >= p.batch) c1 = __ldg(p.chunk_off + p.batch);
    cur.b = b;
    cur.c0 = c0;
    it.b = b;
    it.nch = c1 - c0;
    const int kv = __ldg(p.kv_eff + b);
    it.kv = kv;
    it.q0 = p.q_off != nullptr ? __ldg(p.q_off + b) : b;
    it.qo = p.q_off != nullptr ? __ldg(p.q_len + b) : 1;
    it.tok0 = (it.f - c0) * p.chunk;
    it.tok1 = min(kv, it.tok0 + p.chunk);
    it.ntiles = it.tok1 > it.tok0 && it.qo > 0 ? (it.tok1 - it.tok0 + TK - 1) / TK : 0;
    return it;
}

// Page id of 16-key unit u of an item (-1 past the item's keys) and whether it was loaded
// (a page id inside the pool).  The producers and the Q warps both decide with this, so
// the loads and the softmax's mask agree on which rows of a tile hold data.
__device__ __forceinline__ int unit_page(const Params& p, const Item& it, int u) {
    const int key = it.tok0 + u * PAGE;
    if (key >= it.tok1) return -1;
    return __ldg(p.page_table + (size_t)it.b * p.page_table_stride + key / p.page_size);
}
__device__ __forceinline__ bool page_ok(const Params& p, int pid) {
    return pid >= 0 && pid < p.num_pages;
}

// Exchange of per-warp values among the four warps of a warpgroup through shared memory
// and an mbarrier of count 4 (lane 0 of each warp writes its warp's values, then arrives),
// with a bounded wait: a warp that has given up never leaves the others waiting forever.
// Two areas of 4 x W floats alternate by use, so a warp may write the next exchange while
// a slower one still reads this one (it cannot get two exchanges ahead).  Warp w's values
// come back at out[w * W + i].
struct WgExchange {
    uint32_t bar;
    float* area;   // 2 x 4 x W floats
    uint32_t use;
};
template <int N, int W = 8>
__device__ __forceinline__ bool wg_exchange(WgExchange& x, const float (&vals)[N], int warp4,
                                            int lane, volatile int* abort_flag, int* status,
                                            const float*& out) {
    static_assert(N <= W, "exchange width");
    float* a = x.area + (x.use & 1) * 4 * W;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) a[warp4 * W + i] = vals[i];
        mbar_arrive(x.bar);
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(x.bar, x.use & 1, abort_flag, status));
    ++x.use;
    out = a;
    return ok;
}

// The query rows of an item as the MMA's N = NR columns, column d (thread d of a
// warpgroup), as floats: column n is query row n / G of the item, head g * G + n % G.
// Columns past the item's qo * G rows are zero.
template <int G, int NR>
__device__ __forceinline__ void load_q(const Params& p, const Item& it, int d, float (&qv)[NR]) {
    const int Hq = p.num_qo_heads;
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                             ((size_t)it.q0 * Hq + (size_t)it.g * G) * D + d;
    const int nrows = it.qo * G;
#pragma unroll
    for (int n = 0; n < NR; ++n)
        qv[n] = n < nrows ? __bfloat162float(q[((size_t)(n / G) * Hq + n % G) * D]) : 0.f;
}

// Power-of-two exponent e for the query rows of an item: 2^e * max|q| lies in [2^7, 2^8),
// inside E4M3's range with room for the rounding of hi.  Warpgroup-wide (thread d holds
// column d of the NR rows).
template <int NR>
__device__ __forceinline__ bool q_exponent(const float (&qv)[NR], int d, WgExchange& x,
                                           volatile int* abort_flag, int* status, int& e) {
    float m[1] = {0.f};
#pragma unroll
    for (int h = 0; h < NR; ++h) m[0] = fmaxf(m[0], fabsf(qv[h]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], off));
    const float* a;
    if (!wg_exchange<1>(x, m, d >> 5, d & 31, abort_flag, status, a)) return false;
    const float mm = fmaxf(fmaxf(a[0], a[8]), fmaxf(a[16], a[24]));
    e = 0;
    if (mm > 0.f && mm < INFINITY) {
        const int ex = ((__float_as_int(mm) >> 23) & 0xff) - 127;  // floor(log2 mm), normal
        e = max(-100, min(100, 7 - max(ex, -126)));
    }
    return true;
}

__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// One step of a transposing butterfly over the lanes: N values per lane become N / 2, each
// combined (max or sum) over the lane pair (lane, lane ^ OFF); the lane with bit OFF set
// keeps the upper half.  With N == 1 it is a plain butterfly step.
template <int N, int OFF, bool MAX>
__device__ __forceinline__ void tr_step(float* a, int lane) {
    if constexpr (N >= 2) {
        const bool up = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float keep = up ? a[i + N / 2] : a[i];
            const float send = up ? a[i] : a[i + N / 2];
            const float other = __shfl_xor_sync(0xffffffffu, send, OFF);
            a[i] = MAX ? fmaxf(keep, other) : keep + other;
        }
    } else {
        const float other = __shfl_xor_sync(0xffffffffu, a[0], OFF);
        a[0] = MAX ? fmaxf(a[0], other) : a[0] + other;
    }
}
__host__ __device__ constexpr int at_least_1(int n) { return n > 1 ? n : 1; }
// Max or sum of each of N per-lane values over the warp; afterwards a[0] of lane L holds
// the result for value L / (32 / N).  Every value is summed over the same tree of lane
// pairs whatever N is, so a column's sum does not depend on how many columns there are.
template <int N, bool MAX>
__device__ __forceinline__ void tr_reduce(float (&a)[N], int lane) {
    tr_step<N, 16, MAX>(a, lane);
    tr_step<at_least_1(N / 2), 8, MAX>(a, lane);
    tr_step<at_least_1(N / 4), 4, MAX>(a, lane);
    tr_step<at_least_1(N / 8), 2, MAX>(a, lane);
    tr_step<at_least_1(N / 16), 1, MAX>(a, lane);
}

// wg_exchange for values spread over the lanes as tr_reduce leaves them: lane L holds
// value L / (32 / N) of its warp; warp w's values come back at out[w * W + i].
template <int N, int W>
__device__ __forceinline__ bool wg_exchange_cols(WgExchange& x, float val, int warp4, int lane,
                                                 volatile int* abort_flag, int* status,
                                                 const float*& out) {
    static_assert(N <= W && 32 % N == 0, "exchange width");
    float* a = x.area + (x.use & 1) * 4 * W;
    if (lane % (32 / N) == 0) a[warp4 * W + lane / (32 / N)] = val;
    __syncwarp();
    if (lane == 0) mbar_arrive(x.bar);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(x.bar, x.use & 1, abort_flag, status));
    ++x.use;
    out = a;
    return ok;
}

// Column c of the E4M3 operand(s) for values v[0 .. NR-1], each split into hi + lo, one
// byte per row.  Packed (NR <= 8): one operand, hi of value n in row n and lo in row 8 + n,
// so one MMA takes both; otherwise hi in row n of the operand at op, lo in row n of the
// one at op + OP_BYTES.
template <int NR, bool PACK>
__device__ __forceinline__ void store_col_e4m3(uint8_t* op, int c, const float (&v)[NR]) {
    auto lo_at = [&](int n) -> uint32_t {
        return PACK ? sw128_byte(n + 8, c) : (uint32_t)OP_BYTES + sw128_byte(n, c);
    };
#pragma unroll
    for (int n = 0; n < NR; n += 2) {
        uint32_t h, l;
        e4m3_split2(v[n], n + 1 < NR ? v[n + 1] : 0.f, h, l);
        op[sw128_byte(n, c)] = (uint8_t)h;
        op[lo_at(n)] = (uint8_t)l;
        if (n + 1 < NR) {
            op[sw128_byte(n + 1, c)] = (uint8_t)(h >> 8);
            op[lo_at(n + 1)] = (uint8_t)(l >> 8);
        }
    }
}

// Row r (key r) of the P^T operand with 16 query columns, read MN-major with 32-byte swizzle:
// 32 bytes per key, the hi parts of v[0..15] (N = 0..15) and then their lo parts (N =
// 16..31), each half one 16-byte unit; the two units swap places in rows 4-7 of every 8.
__device__ __forceinline__ void store_row_e4m3_sw32(uint8_t* op, int r, const float (&v)[NH]) {
    uint32_t h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) e4m3_split2(v[2 * k], v[2 * k + 1], h[k], l[k]);
    const uint4 hv = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                h[6] | (h[7] << 16));
    const uint4 lv = make_uint4(l[0] | (l[1] << 16), l[2] | (l[3] << 16), l[4] | (l[5] << 16),
                                l[6] | (l[7] << 16));
    const int sw = (r >> 2) & 1;
    uint4* row = reinterpret_cast<uint4*>(op + 32 * r);
    row[sw] = hv;
    row[sw ^ 1] = lv;
}

// Row r (key r) of the packed P^T operand (NR <= 8 query columns), read MN-major without
// swizzle: 16 bytes per key, the hi parts of v[0..7] (N = 0..7) and their lo parts (N =
// 8..15); columns past NR are zero.
template <int NR>
__device__ __forceinline__ void store_row_e4m3_p16(uint8_t* op, int r, const float (&v)[NR]) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        h[k] = l[k] = 0u;
        if (2 * k < NR) e4m3_split2(v[2 * k], 2 * k + 1 < NR ? v[2 * k + 1] : 0.f, h[k], l[k]);
    }
    reinterpret_cast<uint4*>(op)[r] =
        make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

// G query heads per kv head; NR = the MMA's used N columns: G (one query row per request)
// or 16 (up to 16 / G query rows per request)
template <int G, int NR>
__global__ void __launch_bounds__(THREADS, 1) decode_mma_kernel(const __grid_constant__ Params p) {
    static_assert(NR == G || NR == NH, "query columns");
    static_assert((NR <= 8) == (NR == G), "packed operands exactly for one query row");
    constexpr int XW = NR <= 8 ? 8 : 16;  // width of the softmax exchanges
    // NR <= 8: hi and lo of Q and P^T share one operand (rows n and 8 + n), so one MMA
    // per 32-element step covers both and S^T / O^T column 8 + n holds column n's lo part
    constexpr bool PACK = NR <= 8;
    using L = Layout<PACK>;
    constexpr int RAW_STAGES = L::RAW_STAGES, NPB = L::NPB;
    constexpr uint32_t P_STRIDE = L::P_STRIDE;
    constexpr int OFF_RAW = L::OFF_RAW, OFF_Q = L::OFF_Q, OFF_P = L::OFF_P, OFF_RED = L::OFF_RED,
                  OFF_MASK = L::OFF_MASK, OFF_ITEM = L::OFF_ITEM, OFF_BAR = L::OFF_BAR;
    constexpr int RAW_FULL = L::RAW_FULL, RAW_EMPTY = L::RAW_EMPTY, Q_FULL = L::Q_FULL,
                  Q_EMPTY = L::Q_EMPTY, S_FULL = L::S_FULL, S_EMPTY = L::S_EMPTY,
                  P_FULL = L::P_FULL, PV_LAST = L::PV_LAST, O_EMPTY = L::O_EMPTY,
                  MMA_DRAIN = L::MMA_DRAIN, XCH_Q = L::XCH_Q, XCH_SMX = L::XCH_SMX,
                  NUM_BARS = L::NUM_BARS;
    constexpr uint32_t S_COLS = PACK ? 16u : 32u;  // tensor-memory columns of an S^T tile
    constexpr uint32_t S_REGION = PACK ? 16u * MAX_TILES : 32u * MAX_TILES_ROWS;
    constexpr uint32_t TMEM_O = 2u * S_REGION;
    static_assert(TMEM_O + (PACK ? 16u : 32u) <= (uint32_t)TMEM_COLS, "tensor memory columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    uint32_t* unit_mask = reinterpret_cast<uint32_t*>(smem + OFF_MASK);
    int* qe_words = reinterpret_cast<int*>(smem + OFF_MASK + 64);
    uint32_t* km_words = reinterpret_cast<uint32_t*>(smem + OFF_MASK + 72);  // [2][2]
    // item s's geometry in slot s & 1, written by the Q warps with its Q; ntiles < 0 marks
    // the end of the CTA's items
    Item* items = reinterpret_cast<Item*>(smem + OFF_ITEM);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RAW_STAGES; ++s) {
            mbar_init(BAR(RAW_FULL + s), 1);
            mbar_init(BAR(RAW_EMPTY + s), 1);  // the commit of the tile's MMAs
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(Q_FULL + x), 4);  // one arrival per warp
            // released by the QK MMAs' commit and by the four softmax warps once they have
            // read the item's q exponent and unit mask (which the Q warps write with Q)
            mbar_init(BAR(Q_EMPTY + x), 1 + 4);
            mbar_init(BAR(S_FULL + x), 1);
            mbar_init(BAR(S_EMPTY + x), 4);
        }
        for (int x = 0; x < L::N_PFULL; ++x) mbar_init(BAR(P_FULL + x), 4);
        mbar_init(BAR(PV_LAST), 1);
        mbar_init(BAR(O_EMPTY), 4);
        mbar_init(BAR(MMA_DRAIN), 1);
        mbar_init(BAR(XCH_Q), 4);
        mbar_init(BAR(XCH_SMX), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Q rows and P^T rows NR..15 stay zero: clear every buffer once
    for (int i = threadIdx.x; i < (2 * QP_BYTES + NPB * (int)P_STRIDE) / 16; i += THREADS)
        reinterpret_cast<uint4*>(smem + OFF_Q)[i] = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int Hq = p.num_qo_heads;
    const long long n_items = (long long)__ldg(p.chunk_off + p.batch) * p.num_kv_heads;
    const long long stride = gridDim.x;
    // the producers' walk over the CTA's non-empty items (the Q warps walk the same list and
    // publish each item for the MMA thread and the softmax)
    auto next_item = [&](long long from, Item& out, Cursor& pos) -> long long {
        for (long long k = from; k < n_items; k += stride) {
            out = item_of(p, k, pos);
            if (out.ntiles > 0) return k;
        }
        return -1;
    };

    if (warp == 0 || warp == 2 || warp == 3) {
        // ------------------------------------------------------------ TMA producers
        // Producer w takes ring positions ld with ld % PRODUCERS == w: a warp issues its
        // boxes one lane after another, so several warps keep more boxes in flight.
        const uint32_t pw = warp == 0 ? 0u : (uint32_t)(warp - 1);
        // step order: the K tiles of item s, then the V tiles of item s - 1.  The page ids of
        // an item (at most 64 units of 16 keys: lane l holds units l and l + 32) are read one
        // item ahead, so no page-table read waits in front of a tile's loads.
        uint32_t ld = 0;  // raw tiles issued (ring position)
        bool ok = true;
        auto read_ids = [&](const Item& it, int (&ids)[2]) {
#pragma unroll
            for (int k = 0; k < 2; ++k) ids[k] = unit_page(p, it, lane + 32 * k);
        };
        auto load_tiles = [&](const Item& it, const int (&ids)[2], bool v) {
            for (int t = 0; ok && t < it.ntiles; ++t, ++ld) {
                if (ld % PRODUCERS != pw) continue;
                const int u = t * UNITS + lane;  // this lane's 16-key unit within the item
                const int key = it.tok0 + u * PAGE;
                const int pid = __shfl_sync(0xffffffffu, ids[t >> 2], u & 31);
                const bool in_use = lane < UNITS && key < it.tok1;
                const bool valid = in_use && page_ok(p, pid);
                if (!v && in_use && !valid) atomicOr(p.status, PGQA_DEV_BOUNDS);
                const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
                const uint32_t st = ld % RAW_STAGES;
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(BAR(RAW_EMPTY + st), ((ld / RAW_STAGES) & 1) ^ 1,
                                                  abort_flag, p.status));
                if (!ok) break;
                if (lane == 0) {
                    unit_mask[st] = vmask;
                    mbar_arrive_expect_tx(BAR(RAW_FULL + st), (uint32_t)(__popc(vmask) * PAGE * D));
                }
                __syncwarp();
                if (valid)
                    tma_load_4d(s0 + OFF_RAW + st * RAW_BYTES + lane * PAGE * D,
                                v ? &p.tm_vpages : &p.tm_kpages, BAR(RAW_FULL + st), 0,
                                key % p.page_size, it.g, pid);
            }
        };
        Cursor pos;
        Item prev, it;
        prev.ntiles = 0;
        it.ntiles = 0;
        int ids_prev[2] = {-1, -1}, ids[2] = {-1, -1};
        long long cur = next_item(blockIdx.x, it, pos);
        if (cur >= 0) read_ids(it, ids);
        while (ok && cur >= 0) {
            load_tiles(it, ids, false);
            // read ahead while these K tiles are in flight: the next item's geometry and
            // page ids, used by the next step
            Item ni;
            ni.ntiles = 0;
            int ids_next[2] = {-1, -1};
            const long long nxt = ok ? next_item(cur + stride, ni, pos) : -1;
            if (nxt >= 0) read_ids(ni, ids_next);
            if (ok && prev.ntiles > 0) load_tiles(prev, ids_prev, true);
            prev = it;
            ids_prev[0] = ids[0];
            ids_prev[1] = ids[1];
            it = ni;
            ids[0] = ids_next[0];
            ids[1] = ids_next[1];
            cur = nxt;
        }
        if (ok && prev.ntiles > 0) load_tiles(prev, ids_prev, true);
        if (lane == 0) {
            // copies still in flight (an aborted walk) land before the CTA exits
            const uint32_t first = ld > (uint32_t)RAW_STAGES ? ld - RAW_STAGES : 0;
            for (uint32_t k = first; k < ld; ++k)
                if (k % PRODUCERS == pw)
                    mbar_wait_bounded(BAR(RAW_FULL + k % RAW_STAGES), (k / RAW_STAGES) & 1,
                                      nullptr, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // One thread: a loop in which the whole warp reconverges around each issue costs
        // several hundred cycles per tile more (measured), and this thread is the pace.
        if (lane == 0) {
            // Q.K^T: packed, N = 16 (hi and lo rows in one operand); otherwise N = 32 over
            // the hi and lo operands (rows 0-15 and 16-31), S^T columns n and 16 + n
            constexpr uint32_t IDESC_S = idesc_e4m3_f32(TK, PACK ? NH : 2 * NH, false);
            // P.V: B = P^T MN-major, a row of columns per key, the hi parts then the lo
            // parts: packed, N = 16 (O^T columns n and 8 + n); otherwise N = 32 (O^T
            // columns n and 16 + n)
            constexpr uint32_t IDESC_O = idesc_e4m3_f32(D, PACK ? NH : 2 * NH, true, true);
            uint32_t ld = 0, pt = 0, s = 0;  // ring position, P^T tiles, items
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
                return mbar_wait_bounded(bar, parity, abort_flag, p.status);
            };
            auto qk_tiles = [&](const Item& it) {  // after Q_FULL of item s
                const uint32_t x = s & 1;  // Q buffer and S^T region of item s
                ok = wait(BAR(S_EMPTY + x), ((s >> 1) & 1) ^ 1);
                // B = the Q parts: rows (columns of S^T) of 128 dims, K-major
                const uint64_t qh = sdesc_sw128(s0 + OFF_Q + x * QP_BYTES, 16, 1024);
                for (int t = 0; ok && t < it.ntiles; ++t, ++ld) {
                    const uint32_t st = ld % RAW_STAGES;
                    ok = wait(BAR(RAW_FULL + st), (ld / RAW_STAGES) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    // A = the raw K tile: 128 keys of 128 bytes, K-major; 32 dims per MMA
                    const uint64_t kd = sdesc_sw128(s0 + OFF_RAW + st * RAW_BYTES, 16, 1024);
                    const uint32_t d_tm = tmem_base + S_REGION * x + S_COLS * t;
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)
                        mma_e4m3_ss(d_tm, kd + 2u * k, qh + 2u * k, IDESC_S, k > 0 ? 1u : 0u);
                    mma_commit(BAR(RAW_EMPTY + st));
                }
                if (ok) {
                    mma_commit(BAR(S_FULL + x));
                    mma_commit(BAR(Q_EMPTY + x));
                }
            };
            auto pv_tiles = [&](const Item& it, uint32_t sp) {  // sp: the item's index
                if (sp > 0) ok = wait(BAR(O_EMPTY), (sp - 1) & 1);
                // packed: all of the item's P^T tiles are published at once (P_FULL by item
                // parity); otherwise tile by tile (P_FULL by buffer)
                if (PACK && ok) ok = wait(BAR(P_FULL + (sp & 1)), (sp >> 1) & 1);
                for (int t = 0; ok && t < it.ntiles; ++t, ++ld, ++pt) {
                    const uint32_t st = ld % RAW_STAGES, pb = pt % NPB;
                    ok = (PACK || wait(BAR(P_FULL + pb), (pt / NPB) & 1)) &&
                         wait(BAR(RAW_FULL + st), (ld / RAW_STAGES) & 1);
                    if (!ok) break;
                    // rows past the chunk and rows of units that were not loaded become
                    // zeros (only the last tile of a request, or a bad page id)
                    const int nvalid = min(TK, it.tok1 - (it.tok0 + t * TK));
                    const uint32_t um = unit_mask[st] & 0xffu;
                    if (nvalid < TK || um != 0xffu) {
                        uint4* raw = reinterpret_cast<uint4*>(smem + OFF_RAW + st * RAW_BYTES);
                        for (int row = 0; row < TK; ++row)
                            if (row >= nvalid || !((um >> (row >> 4)) & 1u)) {
#pragma unroll
                                for (int u = 0; u < 8; ++u) raw[row * 8 + u] = make_uint4(0, 0, 0, 0);
                            }
                        fence_async_smem();
                    }
                    tc_fence_after();
                    // A = V^T: the raw V tile read MN-major (a key's 128 dims are one
                    // 128-byte row, 8-key groups 1 KB apart; 32 keys per MMA); B = P^T,
                    // MN-major: packed, a 16-byte row per key without swizzle (8-key core
                    // matrices of 128 bytes, 32 keys = 512 bytes per MMA); otherwise a
                    // 32-byte row per key with 32-byte swizzle (8-key groups 256 bytes
                    // apart, 32 keys = 1 KB per MMA)
                    const uint64_t vd = sdesc_sw128(s0 + OFF_RAW + st * RAW_BYTES, RAW_BYTES, 1024);
                    const uint64_t ph = PACK ? sdesc_plain(s0 + OFF_P + pb * P_STRIDE, 128, 128)
                                             : sdesc_sw32(s0 + OFF_P + pb * P_STRIDE, P_STRIDE, 256);
                    constexpr uint32_t PH_STEP = PACK ? 32u : 64u;  // 16-byte units per MMA
#pragma unroll
                    for (int k = 0; k < TK / 32; ++k)
                        mma_e4m3_ss(tmem_base + TMEM_O, vd + 256u * k, ph + PH_STEP * k, IDESC_O,
                                    (t > 0 || k > 0) ? 1u : 0u);
                    // a P^T buffer is next written for the next item, after that item's
                    // softmax has waited for this item's last P.V (its epilogue), so it
                    // needs no release of its own
                    mma_commit(BAR(RAW_EMPTY + st));
                }
                if (ok) mma_commit(BAR(PV_LAST));
            };
            Item prev;
            prev.ntiles = 0;
            while (ok) {
                ok = wait(BAR(Q_FULL + (s & 1)), (s >> 1) & 1);
                if (!ok) break;
                const Item it = items[s & 1];
                if (it.ntiles < 0) break;
                qk_tiles(it);
                if (ok && prev.ntiles > 0) pv_tiles(prev, s - 1);
                prev = it;
                ++s;
            }
            if (ok && prev.ntiles > 0) pv_tiles(prev, s - 1);
            // every MMA issued has completed before tensor memory is released
            mma_commit(BAR(MMA_DRAIN));
            mbar_wait_bounded(BAR(MMA_DRAIN), 0, nullptr, p.status);
        }
    } else if (warp >= W_Q && warp < W_Q + 4) {
        // ------------------------------------------------------------ Q
        // Per item: its query rows, scaled by 2^e, as the E4M3 hi/lo B operand of Q . K^T
        // (row n = column n of S^T, byte d = dim d, written by thread d), and its loaded
        // units (one bit per 16-key unit, for the softmax's mask).
        const int d = threadIdx.x - 32 * W_Q;  // 0..127
        const int wq = warp - W_Q;
        WgExchange xch{BAR(XCH_Q), red, 0};
        uint32_t s = 0;
        bool ok = true;
        Cursor pos;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
        // the next item with keys; items passed over write their rows here: zeros and
        // lse = -inf for a request of a single empty chunk, nothing for one without rows
        auto next_q = [&](long long from, Item& nx) -> long long {
            for (long long k = from; k < n_items; k += stride) {
                nx = item_of(p, k, pos);
                if (nx.ntiles > 0) return k;
                const int nrows = nx.nch == 1 ? nx.qo * G : 0;
                for (int k2 = d; k2 < nrows * (D / 8); k2 += 128) {
                    const int n = k2 / (D / 8), c = k2 % (D / 8);
                    const size_t row = (size_t)(nx.q0 + n / G) * Hq + nx.g * G + n % G;
                    reinterpret_cast<uint4*>(out + row * D)[c] = make_uint4(0, 0, 0, 0);
                    if (c == 0 && p.lse) p.lse[row] = -INFINITY;
                }
            }
            return -1;
        };
        Item it;
        it.ntiles = 0;
        long long cur = next_q(blockIdx.x, it);
        float qv[NR];
#pragma unroll
        for (int n = 0; n < NR; ++n) qv[n] = 0.f;
        if (cur >= 0) load_q<G, NR>(p, it, d, qv);
        while (ok && cur >= 0) {
            Item ni;
            ni.ntiles = 0;
            const long long nxt = next_q(cur + stride, ni);
            float qn[NR];  // the next item's query rows, loaded while this one is written
#pragma unroll
            for (int n = 0; n < NR; ++n) qn[n] = 0.f;
            if (nxt >= 0) load_q<G, NR>(p, ni, d, qn);
            // unit d < 64 of the item: loaded or not (warps 0 and 1 of the group)
            uint32_t bits = 0;
            if (wq < 2) bits = __ballot_sync(0xffffffffu, page_ok(p, unit_page(p, it, d)));
            const uint32_t x = s & 1;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(Q_EMPTY + x), ((s >> 1) & 1) ^ 1,
                                                           abort_flag, p.status));
            if (!ok) break;
            int e;
            ok = q_exponent<NR>(qv, d, xch, abort_flag, p.status, e);
            if (!ok) break;
            const float sc = exp2i(e);
            float v[NR];
#pragma unroll
            for (int n = 0; n < NR; ++n) v[n] = qv[n] * sc;
            store_col_e4m3<NR, PACK>(smem + OFF_Q + x * QP_BYTES, d, v);
            if (d == 0) {
                qe_words[x] = e;
                items[x] = it;
            }
            if (wq < 2 && lane == 0) km_words[2 * x + wq] = bits;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_FULL + x));
            it = ni;
            ++s;
            cur = nxt;
#pragma unroll
            for (int n = 0; n < NR; ++n) qv[n] = qn[n];
        }
        // the end of the CTA's items, in the next slot once it is free
        if (ok) {
            const uint32_t x = s & 1;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(Q_EMPTY + x), ((s >> 1) & 1) ^ 1,
                                                           abort_flag, p.status));
            if (ok) {
                if (d == 0) items[x].ntiles = -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(Q_FULL + x));
            }
        }
    } else if (warp >= W_SMX && warp < W_SMX + 4) {
        // ------------------------------------------------------------ softmax / epilogue
        // Per item s: (A) its S^T tiles and exact max; (B) the epilogue of item s - 1, whose
        // last P.V completes while (A) runs; (C) its P^T tiles and column sums.  Column n
        // of an S^T tile is query row n / G of the item, head n % G.  With NR = G columns
        // the item's scores stay in registers between (A) and (C); with 16 columns (several
        // query rows) (C) reads them from tensor memory a second time.  Column maxima and
        // sums are reduced over a warp by a transposing butterfly and over the four warps
        // through shared memory; lane n < NR then keeps column n's max and sum.  P^T holds
        // 2^8 exp2(s - max), so the sums l carry the same factor, which 1/l cancels and
        // the lse takes out.
        const int w4 = warp & 3;                                // TMEM lane quarter
        const int r = 32 * w4 + lane;                           // key of a tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * w4) << 16;
        WgExchange xch{BAR(XCH_SMX), red + 64, 0};
        const unsigned long long* kmask = reinterpret_cast<const unsigned long long*>(km_words);
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
        const int cl = lane < NR ? lane : 0;                    // this lane's column
        uint32_t pt = 0, s = 0;  // P^T tiles written, items
        bool ok = true;
        Item prev;
        prev.ntiles = 0;
        float prev_m = 0.f, prev_l = 0.f;  // the previous item's max and sum of column cl
        // (B): wait for item j's last P.V, release O^T, write its outputs
        auto epilogue = [&](const Item& it, uint32_t j, float m_c, float l_c) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(PV_LAST), j & 1, abort_flag,
                                                           p.status));
            if (!ok) return;
            tc_fence_after();
            float ov[NR];  // thread r: column r of O, every query column
            if constexpr (PACK) {  // hi part + lo part
                uint32_t v[16];
                tmem_ld16(tmem_base + lane_base + TMEM_O, v);
                tmem_wait_ld16(v);
#pragma unroll
                for (int n = 0; n < NR; ++n) ov[n] = __uint_as_float(v[n]) + __uint_as_float(v[8 + n]);
            } else {  // columns n (hi part) and 16 + n (lo part)
                uint32_t v[32];
                tmem_ld32(tmem_base + lane_base + TMEM_O, v);
                tmem_wait_ld32(v);
#pragma unroll
                for (int n = 0; n < NR; ++n) ov[n] = __uint_as_float(v[n]) + __uint_as_float(v[NH + n]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(O_EMPTY));
            // lane n < NR: column n's output scale and lse
            const float inv_c = l_c > 0.f ? p.v_scale / l_c : 0.f;
            const float lse_c = l_c > 0.f ? (m_c - P_LOG2_SCALE + log2f(l_c)) * 0.69314718055994531f
                                          : -INFINITY;
            const int nrows = it.qo * G;
#pragma unroll
            for (int n = 0; n < NR; ++n) {
                const float inv = __shfl_sync(0xffffffffu, inv_c, n);
                if (n < nrows) {
                    const int qi = n / G, hq = it.g * G + n % G;
                    const float o = ov[n] * inv;
                    if (it.nch == 1)
                        out[((size_t)(it.q0 + qi) * Hq + hq) * D + r] = __float2bfloat16_rn(o);
                    else
                        p.part_o[(((size_t)it.f * p.max_qo + qi) * Hq + hq) * D + r] = o;
                }
            }
            if (w4 == 0 && lane < NR && lane < nrows) {
                const int qi = lane / G, hq = it.g * G + lane % G;
                if (it.nch == 1) {
                    if (p.lse) p.lse[(size_t)(it.q0 + qi) * Hq + hq] = lse_c;
                } else {
                    p.part_lse[((size_t)it.f * p.max_qo + qi) * Hq + hq] = lse_c;
                }
            }
        };
        while (ok) {
            // (A) the item (published with its Q), the scale of its query rows and its
            // loaded units, then its scores
            const uint32_t x = s & 1;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(Q_FULL + x), (s >> 1) & 1,
                                                           abort_flag, p.status));
            if (!ok) break;
            const Item it = items[x];
            if (it.ntiles < 0) break;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(BAR(S_FULL + x), (s >> 1) & 1,
                                                           abort_flag, p.status));
            if (!ok) break;
            const float c_eff = p.scale_log2 * exp2i(-qe_words[x]);  // score units: log2
            const unsigned long long km = kmask[x];
            // the Q warps may now write the next item of this Q buffer: without this
            // arrival they could complete Q_FULL twice before a slow softmax waits
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_EMPTY + x));
            const uint32_t s_base = tmem_base + lane_base + S_REGION * x;
            tc_fence_after();
            // bit n set: key r of tile t counts for column n (inside the chunk, its unit
            // loaded, and, causal with several query rows, row n / G >= key - (kv - qo))
            auto vis_mask = [&](int t) -> uint32_t {
                const int key = it.tok0 + t * TK + r;
                if (!(key < it.tok1 && ((km >> (8 * t + (r >> 4))) & 1ull))) return 0u;
                if (!p.causal) return 0xFFFFu;
                const int dk = key - (it.kv - it.qo);
                if (dk <= 0) return 0xFFFFu;
                return dk * G >= 16 ? 0u : (0xFFFFu << (dk * G)) & 0xFFFFu;
            };
            float mx[NR];
            float sv[NR == G ? MAX_TILES : 1][NR];  // the item's scores (NR == G only)
            if constexpr (NR == G) {
                // one query row (qo == 1): every score of the item in registers
#pragma unroll
                for (int t = 0; t < MAX_TILES; ++t) {
                    const bool valid = t < it.ntiles && vis_mask(t) != 0u;
                    if (t < it.ntiles) {
                        uint32_t u[16];  // column n: the hi part, column 8 + n: the lo part
                        tmem_ld16(s_base + 16u * t, u);
                        tmem_wait_ld16(u);
#pragma unroll
                        for (int n = 0; n < NR; ++n)
                            sv[t][n] = valid ? (__uint_as_float(u[n]) + __uint_as_float(u[8 + n])) * c_eff
                                             : -INFINITY;
                    } else {
#pragma unroll
                        for (int n = 0; n < NR; ++n) sv[t][n] = -INFINITY;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(S_EMPTY + x));
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    float m = sv[0][n];
#pragma unroll
                    for (int t = 1; t < MAX_TILES; ++t) m = fmaxf(m, sv[t][n]);
                    mx[n] = m;
                }
            } else {
                // 16 columns: a first pass over the tiles for the max (column n of a tile
                // is the hi part, column 16 + n the lo part)
#pragma unroll
                for (int n = 0; n < NR; ++n) mx[n] = -INFINITY;
                const uint64_t c2 = f2_pack(c_eff, c_eff);
                for (int t = 0; t < it.ntiles; ++t) {
                    uint32_t u[32];
                    tmem_ld32(s_base + S_COLS * t, u);
                    tmem_wait_ld32(u);
                    const uint32_t vm = vis_mask(t);
                    float a[NR];  // scores (hi + lo) in log2 units, pairs of columns at once
#pragma unroll
                    for (int n = 0; n < NR; n += 2)
                        f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(u[n]), __uint_as_float(u[n + 1])),
                                                f2_pack(__uint_as_float(u[NH + n]),
                                                        __uint_as_float(u[NH + n + 1]))),
                                         c2),
                                  a[n], a[n + 1]);
                    if (vm == 0xFFFFu) {  // every column sees key r (all but edge tiles)
#pragma unroll
                        for (int n = 0; n < NR; ++n) mx[n] = fmaxf(mx[n], a[n]);
                    } else {
#pragma unroll
                        for (int n = 0; n < NR; ++n)
                            mx[n] = fmaxf(mx[n], ((vm >> n) & 1u) ? a[n] : -INFINITY);
                    }
                }
            }
            // exact max per column over the item's keys
            tr_reduce<NR, true>(mx, lane);
            const float* rt;  // [warp][column]
            ok = wg_exchange_cols<NR, XW>(xch, mx[0], w4, lane, abort_flag, p.status, rt);
            if (!ok) break;
            float neg[NR];  // exp2 offset of column n: 8 - max (P^T = 2^8 exp2(s - max))
#pragma unroll
            for (int n = 0; n < NR; ++n) {
                const float m = fmaxf(fmaxf(rt[n], rt[XW + n]), fmaxf(rt[2 * XW + n], rt[3 * XW + n]));
                neg[n] = (m == -INFINITY ? 0.f : -m) + P_LOG2_SCALE;
            }
            const float m_c =
                fmaxf(fmaxf(rt[cl], rt[XW + cl]), fmaxf(rt[2 * XW + cl], rt[3 * XW + cl]));
            // (B) the previous item's epilogue
            if (prev.ntiles > 0) {
                epilogue(prev, s - 1, prev_m, prev_l);
                if (!ok) break;
            }
            // (C) P^T tiles, E4M3 hi/lo, one buffer per tile (the previous item's last P.V
            // has completed: the epilogue waited for it)
            float l[NR];
#pragma unroll
            for (int n = 0; n < NR; ++n) l[n] = 0.f;
            for (int t = 0; t < it.ntiles; ++t, ++pt) {
                const uint32_t pb = pt % NPB;
                float pv[NR];
                if constexpr (NR == G) {
#pragma unroll
                    for (int tt = 0; tt < MAX_TILES; ++tt) {
                        if (tt == t) {
#pragma unroll
                            for (int n = 0; n < NR; ++n) pv[n] = ex2_approx(sv[tt][n] + neg[n]);
                        }
                    }
                } else {
                    uint32_t u[32];
                    tmem_ld32(s_base + S_COLS * t, u);
                    tmem_wait_ld32(u);
                    const uint32_t vm = vis_mask(t);
                    const uint64_t c2 = f2_pack(c_eff, c_eff);
                    float e[NR];  // exponents: score - max + 8, pairs of columns at once
#pragma unroll
                    for (int n = 0; n < NR; n += 2)
                        f2_unpack(f2_fma(f2_add(f2_pack(__uint_as_float(u[n]), __uint_as_float(u[n + 1])),
                                                f2_pack(__uint_as_float(u[NH + n]),
                                                        __uint_as_float(u[NH + n + 1]))),
                                         c2, f2_pack(neg[n], neg[n + 1])),
                                  e[n], e[n + 1]);
                    if (vm == 0xFFFFu) {  // every column sees key r (all but edge tiles)
#pragma unroll
                        for (int n = 0; n < NR; ++n) pv[n] = ex2_approx(e[n]);
                    } else {
#pragma unroll
                        for (int n = 0; n < NR; ++n) pv[n] = ((vm >> n) & 1u) ? ex2_approx(e[n]) : 0.f;
                    }
                }
#pragma unroll
                for (int n = 0; n < NR; ++n) l[n] += pv[n];
                if constexpr (PACK)
                    store_row_e4m3_p16<NR>(smem + OFF_P + pb * P_STRIDE, r, pv);
                else
                    store_row_e4m3_sw32(smem + OFF_P + pb * P_STRIDE, r, pv);
                if constexpr (!PACK) {
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(P_FULL + pb));
                }
            }
            if (!ok) break;
            if constexpr (PACK) {  // the item's P^T tiles at once
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(P_FULL + (s & 1)));
            }
            if constexpr (NR != G) {  // the second pass has read the item's scores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(S_EMPTY + x));
            }
            // column sums over the item's keys: the warp, then the four warps (read out at
            // once: the exchange area is reused two exchanges later)
            tr_reduce<NR, false>(l, lane);
            const float* rl;
            ok = wg_exchange_cols<NR, XW>(xch, l[0], w4, lane, abort_flag, p.status, rl);
            if (!ok) break;
            prev_l = (rl[cl] + rl[XW + cl]) + (rl[2 * XW + cl] + rl[3 * XW + cl]);
            prev_m = m_c;
            prev = it;
            ++s;
        }
        if (ok && prev.ntiles > 0) epilogue(prev, s - 1, prev_m, prev_l);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int G, int NR>
static cudaError_t launch_g(const Params& p, int num_sms, cudaStream_t stream) {
    static std::atomic<bool> configured[64];  // per device, set once (repeats are harmless)
    constexpr int SMEM_BYTES = Layout<(NR <= 8)>::SMEM_BYTES;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(
            decode_mma_kernel<G, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    decode_mma_kernel<G, NR><<<num_sms, THREADS, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

// one query row per request: G columns; several: all 16 (p.max_qo * G <= 16)
template <int G>
static cudaError_t launch_rows(const Params& p, int num_sms, cudaStream_t stream) {
    if (p.max_qo <= 1) return launch_g<G, G>(p, num_sms, stream);
    if (p.max_qo * G > NH || p.chunk > MAX_TILES_ROWS * TK) return cudaErrorInvalidValue;
    return launch_g<G, NH>(p, num_sms, stream);
}

}  // namespace mmad

// The E4M3 decode on the tensor cores (p.tm_kpages / p.tm_vpages: one-byte 4-D page maps
// with a box of 16 slots of one head; p.scale_log2 carries sm_scale * k_scale * log2 e,
// p.v_scale the value scale).
cudaError_t launch_decode_mma(const Params& p, int group, int num_sms, cudaStream_t stream) {
    switch (group) {
        case 1: return mmad::launch_rows<1>(p, num_sms, stream);
        case 2: return mmad::launch_rows<2>(p, num_sms, stream);
        case 4: return mmad::launch_rows<4>(p, num_sms, stream);
        case 8: return mmad::launch_rows<8>(p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace decode
}  // namespace pgqa
