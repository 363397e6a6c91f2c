// decode.cu -- paged GQA decode (one query row per request) with split-KV and an LSE
// merge, for sm_103a.
//
// What it computes: for request b and query head h, with kv_len keys stored in an NHD
// page table (key j in slot j % page_size of page page_table[b][j / page_size]),
//   o[b,h] = softmax_j(sm_scale * q[b,h] . k[j, h/G]) v[j, h/G],
//   lse[b,h] = ln sum_j exp(sm_scale * q[b,h] . k[j, h/G]).
// Sources: vllm-rlt pull request "feat: add FlashInfer attention backend for SM120
// decode" (Scope and Design notes: paged decode over a block table, block size 16,
// kv_layout "NHD", padding in the table never visible, zero-length rows give zeros);
// FlashInfer documentation, flashinfer.cascade "Merge Attention States" (how partial
// results over disjoint key sets combine).
//
// Design: with bf16 K/V the path is bound by HBM bandwidth (about 4 flops per KV byte), so
// it runs on the CUDA cores, not the tensor cores.  (An E4M3 cache takes the tensor-core
// decode of decode_mma.cu, which shares this file's plan and merge kernels.)
//  * plan_kernel: sanitises kv_lens and cuts each request into chunks of `chunk` keys
//    (1024, or 512 / 256 / 128 for calls with little work; chosen from the call's shape).
//    For a given chunk length the cut depends on the request alone, so a request's
//    result does not depend on what else is in the batch.
//  * decode_tma_kernel: one warp per (chunk, kv head).  Pages stream through a per-warp
//    TMA ring in shared memory; the online softmax keeps a running max and sum per
//    head.  A request with a single chunk writes its bf16 output directly; otherwise
//    each chunk writes a normalised fp32 partial output and its lse.
//  * merge_kernel: each (request, head) with more than one chunk combines the partials
//    with weights exp(lse_c - max lse), in groups of 8 chunks; a warp per row, or a CTA
//    per row when there are few rows (same arithmetic, same order).
#include <atomic>

#include "ptx.cuh"

namespace pgqa {
namespace decode {

// ---------------------------------------------------------------------------- plan
__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(PlanParams p) {
    __shared__ int scan[PLAN_THREADS];
    const int tid = threadIdx.x, nthr = blockDim.x;
    int running = 0;
    for (int base = 0; base < p.batch; base += nthr) {
        const int b = base + tid;
        int cnt = 0;
        if (b < p.batch) {
            int n = p.kv_lens[b];
            if (n < 0 || n > p.max_kv) {
                atomicOr(p.status, PGQA_DEV_BOUNDS);
                n = 0;
            }
            if (p.q_indptr != nullptr) {
                // a request with a bad query range keeps no keys and no rows: nothing of it
                // is computed or written
                const int q0 = p.q_indptr[b], qo = p.q_indptr[b + 1] - q0;
                const bool q_ok = q0 >= 0 && qo >= 0 && qo <= p.max_qo;
                if (!q_ok) {
                    atomicOr(p.status, PGQA_DEV_BOUNDS);
                    n = 0;
                }
                p.q_off[b] = q_ok ? q0 : 0;
                p.q_len[b] = q_ok ? qo : 0;
            }
            p.kv_eff[b] = n;
            cnt = n > 0 ? (n + p.chunk - 1) / p.chunk : 1;
        }
        scan[tid] = cnt;
        __syncthreads();
        for (int off = 1; off < nthr; off <<= 1) {
            const int v = tid >= off ? scan[tid - off] : 0;
            __syncthreads();
            scan[tid] += v;
            __syncthreads();
        }
        if (b < p.batch) p.chunk_off[b] = running + scan[tid] - cnt;
        running += scan[nthr - 1];
        __syncthreads();
    }
    if (tid == 0) p.chunk_off[p.batch] = running;
}

__device__ __forceinline__ int find_request(const int* off, int batch, int f) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(off + mid) <= f) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// One butterfly step of the transposing reduction: N values per lane become N/2, each
// the sum over the lane pair (lane, lane ^ OFF); the lane with bit OFF set keeps the
// upper half.  With N == 1 it is a plain butterfly add.
template <int N, int OFF>
__device__ __forceinline__ void tr_step(float* a, int lane) {
    if constexpr (N >= 2) {
        const bool up = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float keep = up ? a[i + N / 2] : a[i];
            const float send = up ? a[i] : a[i + N / 2];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
        }
    } else {
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], OFF);
    }
}

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Sum N = 16 * G per-lane partial values over the 32 lanes.  Afterwards lane L holds
// VPL = max(1, N / 32) full sums: value index v = L * VPL + x for N >= 32, v = L / 2 for
// N == 16 (lanes 2v and 2v+1 then hold the same sum).
template <int N>
__device__ __forceinline__ void transpose_reduce(float* a, int lane) {
    tr_step<N, 16>(a, lane);
    tr_step<cmax(N / 2, 1), 8>(a, lane);
    tr_step<cmax(N / 4, 1), 4>(a, lane);
    tr_step<cmax(N / 8, 1), 2>(a, lane);
    tr_step<cmax(N / 16, 1), 1>(a, lane);
}

// ------------------------------------------------------------ TMA-staged decode
// One warp per (chunk, kv head) item.  The warp streams its keys in units of 16 tokens
// (one page of 16, or a 16-token slice of a larger page) with TMA (one 4 KB box per unit
// for K and one for V) into a private two-stage ring in shared memory; lane 0
// issues the copies and refills a stage as soon as the warp has finished reading it.
// Lane (tp, ds) = (lane / 16, lane % 16) works on head-dim elements 8*ds .. 8*ds+7 of
// the page's tokens with parity tp: 16-byte shared-memory reads of two whole K (V) rows
// per warp instruction, packed f32x2 FMAs, and a transposing reduction of the 8*G
// partial dot products over the 16 lanes of a parity (30 shuffles for G = 4).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// 8 bf16 -> 4 packed fp32 pairs (element 2k in the low half of pair k)
__device__ __forceinline__ void bf16x8_to_pairs(const uint4& r, uint64_t (&o)[4]) {
    o[0] = f2_pack(bf_lo(r.x), bf_hi(r.x));
    o[1] = f2_pack(bf_lo(r.y), bf_hi(r.y));
    o[2] = f2_pack(bf_lo(r.z), bf_hi(r.z));
    o[3] = f2_pack(bf_lo(r.w), bf_hi(r.w));
}

template <int G>
__global__ void __launch_bounds__(WARPS * 32, G >= 8 ? 2 : 3)
    decode_tma_kernel(const __grid_constant__ Params p) {
    constexpr int D = HEAD_DIM;
    constexpr int UNIT = PAGE * D * 2;           // one 16-token unit of one head (bf16)
    constexpr int NST = STAGES;
    constexpr int SB = 2 * UNIT;                 // K + V of a unit
    static_assert(NST * SB == STAGES * STAGE_BYTES, "ring size");
    constexpr int NV = 8 * G;                     // partial dot products per lane per page
    constexpr int VPL = NV >= 16 ? NV / 16 : 1;   // full scores per lane after the reduction
    constexpr int GS = 16 / G;                    // d-slices per head among the score lanes
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int tp = lane >> 4, ds = lane & 15;
    uint8_t* wsm = smem + wib * WARP_SMEM;
    const uint32_t stage0 = smem_u32(wsm);
    float* ps = reinterpret_cast<float*>(wsm + NST * SB);  // [16 tokens][G]
    const uint32_t full0 = smem_u32(wsm + NST * SB + 512);
    if (lane == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(full0 + 8 * s, 1);
        fence_barrier_init();
    }
    __syncwarp();

    const int Hq = p.num_qo_heads, Hk = p.num_kv_heads;
    const int total_chunks = __ldg(p.chunk_off + p.batch);
    const long long n_items = (long long)total_chunks * Hk;

    // head / token of each score this lane holds after the reduction
    int my_h[VPL], my_i[VPL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
        const int v = NV >= 16 ? ds * VPL + x : ds >> 1;
        my_h[x] = v / 8;
        my_i[x] = v % 8;
    }
    const int head_of_lane = my_h[0];
    const bool dup_lane = NV < 16 && (ds & 1);
    uint32_t issued = 0, consumed = 0;  // pages this warp loaded / used (ring position)
    bool ok = true;

    for (long long item = (long long)blockIdx.x * WARPS + wib; ok && item < n_items;
         item += (long long)gridDim.x * WARPS) {
        const int f = (int)(item / Hk);
        const int g = (int)(item % Hk);
        const int b = find_request(p.chunk_off, p.batch, f);
        const int c = f - __ldg(p.chunk_off + b);
        const int nch = __ldg(p.chunk_off + b + 1) - __ldg(p.chunk_off + b);
        const int kv_len = __ldg(p.kv_eff + b);
        const int tok0 = c * p.chunk;
        const int tok1 = min(kv_len, tok0 + p.chunk);
        const int page0 = tok0 / PAGE;  // first 16-token unit of the chunk
        const int np = (tok1 - tok0 + PAGE - 1) / PAGE;
        const int* pt_row = p.page_table + (size_t)b * p.page_table_stride;
        const int page_size = p.page_size;
        // page id and first slot of 16-token unit u; false if the id is outside the pool
        auto unit_row = [&](int u, int& pid, int& slot) -> bool {
            const int tok = u * PAGE;
            pid = __ldg(pt_row + tok / page_size);
            slot = tok % page_size;
            return pid >= 0 && pid < p.num_pages;
        };

        auto issue = [&](int page) {  // lane 0 only
            int pid, slot;
            const bool valid = unit_row(page, pid, slot);
            const uint32_t st = issued % NST;
            const uint32_t bar = full0 + 8 * st;
            if (valid) {
                mbar_arrive_expect_tx(bar, SB);
                const uint32_t dst = stage0 + st * SB;
                tma_load_4d(dst, &p.tm_kpages, bar, 0, slot, g, pid);
                tma_load_4d(dst + UNIT, &p.tm_vpages, bar, 0, slot, g, pid);
            } else {
                atomicOr(p.status, PGQA_DEV_BOUNDS);
                mbar_arrive(bar);  // the page is skipped; keep the ring in phase
            }
        };
        const int prime = min(np, NST);
        for (int k = 0; k < prime; ++k) {
            if (lane == 0) issue(page0 + k);
            ++issued;
        }

        uint64_t q2[G][4];
        {
            const uint4* qp = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * Hq + g * G) * D);
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                uint64_t t[4];
                bf16x8_to_pairs(__ldg(qp + h * (D / 8) + ds), t);
#pragma unroll
                for (int e = 0; e < 4; ++e) q2[h][e] = f2_mul(t[e], sc2);
            }
        }
        uint64_t o2[G][4];
        float m[G];
        const uint64_t zero2 = f2_pack(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) o2[h][e] = zero2;
        }
        float lp = 0.f;

        for (int pi = 0; pi < np; ++pi) {
            const uint32_t st = consumed % NST;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, (consumed / NST) & 1,
                                                           nullptr, p.status));
            if (!ok) break;
            ++consumed;
            const int page = page0 + pi;
            int pid, slot;
            const int nvalid = unit_row(page, pid, slot) ? min(PAGE, tok1 - page * PAGE) : 0;
            const uint32_t kbase = stage0 + st * SB + ds * 16;
            const uint32_t vbase = kbase + UNIT;

            float part[NV];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint64_t k2[4];
                bf16x8_to_pairs(lds128(kbase + (2 * i + tp) * (D * 2)), k2);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    uint64_t acc = f2_mul(q2[h][0], k2[0]);
                    acc = f2_fma(q2[h][1], k2[1], acc);
                    acc = f2_fma(q2[h][2], k2[2], acc);
                    acc = f2_fma(q2[h][3], k2[3], acc);
                    float a0, a1;
                    f2_unpack(acc, a0, a1);
                    part[h * 8 + i] = a0 + a1;
                }
            }
            tr_step<NV, 8>(part, lane);
            tr_step<cmax(NV / 2, 1), 4>(part, lane);
            tr_step<cmax(NV / 4, 1), 2>(part, lane);
            tr_step<cmax(NV / 8, 1), 1>(part, lane);

            float sc[VPL];
            float gmax = -INFINITY;
#pragma unroll
            for (int x = 0; x < VPL; ++x) {
                sc[x] = 2 * my_i[x] + tp < nvalid ? part[x] : -INFINITY;
                gmax = fmaxf(gmax, sc[x]);
            }
#pragma unroll
            for (int off = 1; off < GS; off <<= 1)
                gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
            gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, 16));
            float alpha[G];
            float m_use_mine = 0.f, alpha_mine = 1.f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pm = __shfl_sync(0xffffffffu, gmax, h * GS);
                const float m_new = fmaxf(m[h], pm);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha[h] = ex2_approx(m[h] - m_use);
                m[h] = m_new;
                if (h == head_of_lane) {
                    m_use_mine = m_use;
                    alpha_mine = alpha[h];
                }
            }
            float psum = 0.f;
#pragma unroll
            for (int x = 0; x < VPL; ++x) {
                const float pv = ex2_approx(sc[x] - m_use_mine);
                psum += pv;
                ps[(2 * my_i[x] + tp) * G + my_h[x]] = pv;
            }
            lp = lp * alpha_mine + (dup_lane ? 0.f : psum);
            __syncwarp();
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint64_t a2 = f2_pack(alpha[h], alpha[h]);
#pragma unroll
                for (int e = 0; e < 4; ++e) o2[h][e] = f2_mul(o2[h][e], a2);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = 2 * i + tp;
                uint64_t v2[4];
                bf16x8_to_pairs(lds128(vbase + t * (D * 2)), v2);
                if (nvalid < PAGE && t >= nvalid) {  // slots past kv_len may hold anything
#pragma unroll
                    for (int e = 0; e < 4; ++e) v2[e] = zero2;
                }
                float pr[G];
                if constexpr (G % 4 == 0) {
#pragma unroll
                    for (int h4 = 0; h4 < G; h4 += 4) {
                        const float4 w = *reinterpret_cast<const float4*>(ps + t * G + h4);
                        pr[h4] = w.x;
                        pr[h4 + 1] = w.y;
                        pr[h4 + 2] = w.z;
                        pr[h4 + 3] = w.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h) pr[h] = ps[t * G + h];
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const uint64_t pp = f2_pack(pr[h], pr[h]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o2[h][e] = f2_fma(pp, v2[e], o2[h][e]);
                }
            }
            __syncwarp();  // every lane is done with this stage and with ps
            if (pi + NST < np) {
                if (lane == 0) {
                    fence_async_smem();
                    issue(page0 + pi + NST);
                }
                ++issued;
            }
        }
        if (!ok) break;

        // the two token parities hold partial sums of the same outputs: combine them
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o2[h][e] = f2_add(o2[h][e], __shfl_xor_sync(0xffffffffu, o2[h][e], 16));
        float lsum = lp;
#pragma unroll
        for (int off = 1; off < GS; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float l = __shfl_sync(0xffffffffu, lsum, h * GS);
            const float inv = l > 0.f ? p.v_scale / l : 0.f;  // v_scale = 1 for bf16 K/V
            const float lse_v = l > 0.f ? (m[h] + log2f(l)) * 0.69314718055994531f : -INFINITY;
            const int hq = g * G + h;
            float o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) f2_unpack(o2[h][e], o[2 * e], o[2 * e + 1]);
            if (tp == 0) {
                if (nch == 1) {
                    uint4 u;
                    u.x = pack_bf16x2(o[0] * inv, o[1] * inv);
                    u.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                    u.z = pack_bf16x2(o[4] * inv, o[5] * inv);
                    u.w = pack_bf16x2(o[6] * inv, o[7] * inv);
                    reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                             ((size_t)b * Hq + hq) * D)[ds] = u;
                } else {
                    float4* op = reinterpret_cast<float4*>(p.part_o + ((size_t)f * Hq + hq) * D);
                    op[2 * ds] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
                    op[2 * ds + 1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
                }
            }
            if (lane == 0) {
                if (nch == 1) {
                    if (p.lse) p.lse[(size_t)b * Hq + hq] = lse_v;
                } else {
                    p.part_lse[(size_t)f * Hq + hq] = lse_v;
                }
            }
        }
    }
    // copies still in flight (an aborted item) land before the warp exits
    while (consumed < issued) {
        mbar_wait_bounded(full0 + 8 * (consumed % NST), (consumed / NST) & 1, nullptr,
                          p.status);
        ++consumed;
    }
}

// One warp per (request, head) row whose request was split into several chunks.
// Merge of one (request, head) row's chunk partials, in a fixed order: chunks are summed
// in groups of MERGE_GROUP consecutive chunks (weights exp(lse_c - max lse)), and the group
// sums are added in group order.  With few rows a whole CTA works on one row (warp w
// computes groups w, w + 8, ...); with many rows one warp computes every group of its row.
// Both do the same floating-point operations in the same order, so the result does not
// depend on which one ran, and so not on the rest of the batch.
constexpr int MERGE_GROUP = 8;
constexpr int MERGE_WARPS = 8;

struct MergeRow {
    int b, i, h, f0, nch;  // request, its query row i, head, first chunk, chunks
    int orow;              // output row
};

// one group's weighted sum (lane: 4 of the D columns) and weight sum
__device__ __forceinline__ void merge_group(const Params& p, const MergeRow& r, int g, float mx,
                                            int lane, float4& acc, float& wsum) {
    constexpr int D = HEAD_DIM;
    const int Hq = p.num_qo_heads;
    const int c0 = g * MERGE_GROUP;
    const int n = min(MERGE_GROUP, r.nch - c0);
    const size_t qh = (size_t)p.max_qo * Hq;   // partial slots per chunk
    const size_t s0 = (size_t)(r.f0 + c0) * qh + (size_t)r.i * Hq + r.h;
    const float* lp = p.part_lse + s0;
    const float4* vp = reinterpret_cast<const float4*>(p.part_o + s0 * D) + lane;
    const size_t vstride = qh * D / 4;  // float4s from one chunk's row to the next
    float l[MERGE_GROUP];
    float4 v[MERGE_GROUP];
#pragma unroll
    for (int u = 0; u < MERGE_GROUP; ++u) {  // every load of the group before any arithmetic
        if (u < n) {
            l[u] = lp[(size_t)u * qh];
            v[u] = vp[(size_t)u * vstride];
        }
    }
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    wsum = 0.f;
#pragma unroll
    for (int u = 0; u < MERGE_GROUP; ++u) {
        if (u < n) {
            const float w = __expf(l[u] - mx);
            wsum += w;
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
    }
}

__device__ __forceinline__ void merge_store(const Params& p, const MergeRow& r, int lane,
                                            float mx, const float4& acc, float wsum) {
    constexpr int D = HEAD_DIM;
    const int Hq = p.num_qo_heads;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)r.orow * Hq + r.h) * D;
    uint2 u;
    u.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    u.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(op + lane * 4) = u;
    if (lane == 0 && p.lse)
        p.lse[(size_t)r.orow * Hq + r.h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

__device__ __forceinline__ float4 f4_add(const float4& a, const float4& b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// SPLIT = false: one warp per row, 8 rows per CTA.  SPLIT = true: one CTA per row.
template <bool SPLIT>
__global__ void __launch_bounds__(MERGE_WARPS * 32) merge_kernel(const Params p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Hq = p.num_qo_heads;
    const long long row = SPLIT ? (long long)blockIdx.x : (long long)blockIdx.x * MERGE_WARPS + warp;
    const long long qh = (long long)p.max_qo * Hq;
    if (row >= (long long)p.batch * qh) return;  // uniform per CTA when SPLIT
    MergeRow r;
    r.b = (int)(row / qh);
    r.i = (int)((row % qh) / Hq);
    r.h = (int)(row % Hq);
    if (p.q_off != nullptr && r.i >= __ldg(p.q_len + r.b)) return;  // no such query row
    r.orow = p.q_off != nullptr ? __ldg(p.q_off + r.b) + r.i : r.b;
    r.f0 = __ldg(p.chunk_off + r.b);
    r.nch = __ldg(p.chunk_off + r.b + 1) - r.f0;
    if (r.nch <= 1) return;  // written by the decode kernel
    const int ngroups = (r.nch + MERGE_GROUP - 1) / MERGE_GROUP;
    // the largest chunk lse
    const int t0 = SPLIT ? warp * 32 + lane : lane, tstep = SPLIT ? MERGE_WARPS * 32 : 32;
    float mx = -INFINITY;
    for (int c = t0; c < r.nch; c += tstep)
        mx = fmaxf(mx, p.part_lse[(size_t)(r.f0 + c) * qh + (size_t)r.i * Hq + r.h]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if constexpr (SPLIT) {
        __shared__ float s_mx[MERGE_WARPS];
        __shared__ float4 s_acc[MERGE_WARPS][32];
        __shared__ float s_w[MERGE_WARPS];
        if (lane == 0) s_mx[warp] = mx;
        __syncthreads();
        mx = s_mx[0];
#pragma unroll
        for (int w = 1; w < MERGE_WARPS; ++w) mx = fmaxf(mx, s_mx[w]);
        float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
        float wtot = 0.f;
        if (mx != -INFINITY) {
            for (int g0 = 0; g0 < ngroups; g0 += MERGE_WARPS) {
                const int g = g0 + warp;
                if (g < ngroups) {
                    float4 acc;
                    float ws;
                    merge_group(p, r, g, mx, lane, acc, ws);
                    s_acc[warp][lane] = acc;
                    if (lane == 0) s_w[warp] = ws;
                }
                __syncthreads();
                if (warp == 0) {  // group sums in group order
                    const int n = min(MERGE_WARPS, ngroups - g0);
                    for (int w = 0; w < n; ++w) {
                        tot = f4_add(tot, s_acc[w][lane]);
                        wtot += s_w[w];
                    }
                }
                __syncthreads();
            }
        }
        if (warp == 0) merge_store(p, r, lane, mx, tot, wtot);
    } else {
        float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
        float wtot = 0.f;
        if (mx != -INFINITY) {
            for (int g = 0; g < ngroups; ++g) {
                float4 acc;
                float ws;
                merge_group(p, r, g, mx, lane, acc, ws);
                tot = f4_add(tot, acc);
                wtot += ws;
            }
        }
        merge_store(p, r, lane, mx, tot, wtot);
    }
}

// ------------------------------------------------------------------ host launchers
cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream) {
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(pp);
    return cudaGetLastError();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor maps over the paged K and V caches as 4-D tensors {d, slot, head, page} with
// element strides slot_stride / head_stride / page_stride (d contiguous); one box is 16
// slots of one kv head (PAGE rows x D elements, 4 KB).
cudaError_t prepare_page_maps(Params& p, const void* k_pages, const void* v_pages,
                              int num_pages, int num_kv_heads, int page_size,
                              long long page_stride, long long slot_stride,
                              long long head_stride, bool kv8) {
    const int eb = kv8 ? 1 : 2;  // bytes per element
    // resolved once; a function-local static is initialised exactly once even when the
    // main entry points and the allocation-free one (different locks) race to first use
    static const EncodeTiledFn encode = []() -> EncodeTiledFn {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn,
                                                               12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(fn);
    }();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[4] = {(cuuint64_t)HEAD_DIM, (cuuint64_t)page_size,
                                (cuuint64_t)num_kv_heads, (cuuint64_t)(num_pages > 0 ? num_pages : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)slot_stride * eb, (cuuint64_t)head_stride * eb,
                                   (cuuint64_t)page_stride * eb};
    const cuuint32_t box[4] = {HEAD_DIM, PAGE, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMap* maps[2] = {&p.tm_kpages, &p.tm_vpages};
    const void* bases[2] = {k_pages, v_pages};
    const CUtensorMapDataType dt = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // E4M3 tiles feed the tensor-core decode, whose converters read them 128-byte swizzled
    const CUtensorMapSwizzle sw = kv8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    for (int i = 0; i < 2; ++i) {
        CUresult r = encode(maps[i], dt, 4, const_cast<void*>(bases[i]),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int G>
static cudaError_t launch_decode_g(const Params& p, int num_sms, cudaStream_t stream) {
    // per device, set up on first use; the entries are atomics because the main entry
    // points and the allocation-free one hold different locks (a repeated set-up is
    // harmless: it computes the same value)
    static std::atomic<int> blocks_per_sm[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int bps = blocks_per_sm[dev].load(std::memory_order_acquire);
    if (bps == 0) {
        cudaError_t e = cudaFuncSetAttribute(decode_tma_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tma_kernel<G>, WARPS * 32,
                                                          SMEM_BYTES);
        if (e != cudaSuccess) return e;
        bps = n > 0 ? n : 1;
        blocks_per_sm[dev].store(bps, std::memory_order_release);
    }
    const int grid = num_sms * bps;
    decode_tma_kernel<G><<<grid, WARPS * 32, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

// bf16 K/V pages (the E4M3 decode runs on the tensor cores: decode_mma.cu)
cudaError_t launch_decode(const Params& p, int group, int num_sms, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_decode_g<1>(p, num_sms, stream);
        case 2: return launch_decode_g<2>(p, num_sms, stream);
        case 4: return launch_decode_g<4>(p, num_sms, stream);
        case 8: return launch_decode_g<8>(p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const Params& p, cudaStream_t stream) {
    const long long rows = (long long)p.batch * p.max_qo * p.num_qo_heads;
    if (rows <= 0) return cudaSuccess;
    // too few rows to fill the GPU with one warp per row: a CTA per row (the result is
    // the same bits either way)
    if (rows < 1024)
        merge_kernel<true><<<(unsigned)rows, MERGE_WARPS * 32, 0, stream>>>(p);
    else
        merge_kernel<false><<<(unsigned)((rows + MERGE_WARPS - 1) / MERGE_WARPS),
                              MERGE_WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace decode
}  // namespace pgqa
