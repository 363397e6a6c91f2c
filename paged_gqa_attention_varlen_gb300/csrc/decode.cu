// decode.cu -- paged GQA decode (one query row per request) with split-KV and an LSE
// merge, for sm_103a.
//
// What it computes: for request b and query head h, with kv_len keys stored in an NHD
// page table (key j in slot j % 16 of page page_table[b][j / 16]),
//   o[b,h] = softmax_j(sm_scale * q[b,h] . k[j, h/G]) v[j, h/G],
//   lse[b,h] = ln sum_j exp(sm_scale * q[b,h] . k[j, h/G]).
// Sources: vllm-rlt pull request "feat: add FlashInfer attention backend for SM120
// decode" (Scope and Design notes: paged decode over a block table, block size 16,
// kv_layout "NHD", padding in the table never visible, zero-length rows give zeros);
// FlashInfer documentation, flashinfer.cascade "Merge Attention States" (how partial
// results over disjoint key sets combine).
//
// Design: the path is bound by HBM bandwidth (about 4 flops per KV byte), so it runs on
// the CUDA cores, not the tensor cores.
//  * plan_kernel: sanitises kv_lens and cuts each request into chunks of CHUNK keys.
//    The cut depends on the request alone, so a request's result does not depend on
//    what else is in the batch.
//  * decode_kernel: one warp per (chunk, kv head).  Lane i holds head_dim elements
//    4i..4i+3 of the G query heads; each page's 16 K rows and 16 V rows are fetched
//    with 8-byte loads (a 256-byte row per warp instruction), the next page's rows are
//    prefetched into registers while the current page is computed, the G x 16 partial
//    dot products are reduced across lanes by a transposing butterfly (62 shuffles for
//    G = 4), and the online softmax keeps a running max and sum per head.  A request
//    with a single chunk writes its bf16 output directly; otherwise each chunk writes a
//    normalised fp32 partial output and its lse.
//  * merge_kernel: one warp per (request, head) with more than one chunk combines the
//    partials with weights exp(lse_c - max lse).
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
            p.kv_eff[b] = n;
            cnt = n > 0 ? (n + CHUNK - 1) / CHUNK : 1;
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

__device__ __forceinline__ uint2 ldg_nc_v2(const void* ptr) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(ptr));
    return r;
}

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

template <int G>
__global__ void __launch_bounds__(WARPS * 32) decode_kernel(const Params p) {
    constexpr int D = HEAD_DIM;
    constexpr int NV = 16 * G;                       // scores per page
    constexpr int VPL = NV >= 32 ? NV / 32 : 1;      // scores held per lane after reduction
    constexpr int GS = 32 / G;                       // lanes holding one head's scores
    __shared__ float ps_all[WARPS][16 * G];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    float* ps = ps_all[wib];
    const int Hq = p.num_qo_heads, Hk = p.num_kv_heads;
    const int total_chunks = __ldg(p.chunk_off + p.batch);
    const long long n_items = (long long)total_chunks * Hk;
    const long long row_stride = (long long)Hk * D;  // elements between consecutive slots
    const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(p.k_pages);
    const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(p.v_pages);

    // head / token of each score this lane holds after the reduction
    int my_h[VPL], my_t[VPL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
        const int v = NV >= 32 ? lane * VPL + x : lane >> 1;
        my_h[x] = v / 16;
        my_t[x] = v % 16;
    }
    const int head_of_lane = my_h[0];
    const bool dup_lane = NV < 32 && (lane & 1);

    for (long long item = (long long)blockIdx.x * WARPS + wib; item < n_items;
         item += (long long)gridDim.x * WARPS) {
        const int f = (int)(item / Hk);
        const int g = (int)(item % Hk);
        const int b = find_request(p.chunk_off, p.batch, f);
        const int c = f - __ldg(p.chunk_off + b);
        const int nch = __ldg(p.chunk_off + b + 1) - __ldg(p.chunk_off + b);
        const int kv_len = __ldg(p.kv_eff + b);
        const int tok0 = c * CHUNK;
        const int tok1 = min(kv_len, tok0 + CHUNK);

        float q[G][4];
        {
            const uint2* qp = reinterpret_cast<const uint2*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * Hq + g * G) * D);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint2 u = __ldg(qp + h * (D / 4) + lane);
                q[h][0] = bf_lo(u.x) * p.scale_log2;
                q[h][1] = bf_hi(u.x) * p.scale_log2;
                q[h][2] = bf_lo(u.y) * p.scale_log2;
                q[h][3] = bf_hi(u.y) * p.scale_log2;
            }
        }
        float o[G][4];
        float m[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] = 0.f;
        }
        float lp = 0.f;

        const int page0 = tok0 / PAGE;
        const int page1 = (tok1 + PAGE - 1) / PAGE;  // exclusive
        const int* pt_row = p.page_table + (size_t)b * p.page_table_stride;

        uint2 kr[16], vr[16];
        auto load_page = [&](int page) {
            int pid = __ldg(pt_row + page);
            const bool ok = pid >= 0 && pid < p.num_pages;
            if (!ok && lane == 0) atomicOr(p.status, PGQA_DEV_BOUNDS);
            const int base_tok = page * PAGE;
            const size_t base = ((size_t)(ok ? pid : 0) * PAGE * Hk + g) * D + lane * 4;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const bool valid = ok && (base_tok + t < tok1);
                kr[t] = valid ? ldg_nc_v2(kp + base + t * row_stride) : make_uint2(0, 0);
                vr[t] = valid ? ldg_nc_v2(vp + base + t * row_stride) : make_uint2(0, 0);
            }
        };
        if (page0 < page1) load_page(page0);
        for (int page = page0; page < page1; ++page) {
            uint2 kc[16], vc[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                kc[t] = kr[t];
                vc[t] = vr[t];
            }
            if (page + 1 < page1) load_page(page + 1);
            const int base_tok = page * PAGE;

            float part[NV];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float k0 = bf_lo(kc[t].x), k1 = bf_hi(kc[t].x);
                const float k2 = bf_lo(kc[t].y), k3 = bf_hi(kc[t].y);
#pragma unroll
                for (int h = 0; h < G; ++h)
                    part[h * 16 + t] = fmaf(q[h][0], k0, fmaf(q[h][1], k1,
                                            fmaf(q[h][2], k2, q[h][3] * k3)));
            }
            transpose_reduce<NV>(part, lane);

            float sc[VPL];
            float gmax = -INFINITY;
#pragma unroll
            for (int x = 0; x < VPL; ++x) {
                const bool valid = base_tok + my_t[x] < tok1;
                sc[x] = valid ? part[x] : -INFINITY;
                gmax = fmaxf(gmax, sc[x]);
            }
#pragma unroll
            for (int off = GS / 2; off >= 1; off >>= 1)
                gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
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
                ps[my_t[x] * G + my_h[x]] = pv;
            }
            lp = lp * alpha_mine + (dup_lane ? 0.f : psum);
            __syncwarp();
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[h][e] *= alpha[h];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float v0 = bf_lo(vc[t].x), v1 = bf_hi(vc[t].x);
                const float v2 = bf_lo(vc[t].y), v3 = bf_hi(vc[t].y);
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
                    o[h][0] = fmaf(pr[h], v0, o[h][0]);
                    o[h][1] = fmaf(pr[h], v1, o[h][1]);
                    o[h][2] = fmaf(pr[h], v2, o[h][2]);
                    o[h][3] = fmaf(pr[h], v3, o[h][3]);
                }
            }
            __syncwarp();
        }

        // finish: per-head sums, normalise, write
        float lsum = lp;
#pragma unroll
        for (int off = GS / 2; off >= 1; off >>= 1)
            lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float l = __shfl_sync(0xffffffffu, lsum, h * GS);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse_v = l > 0.f ? (m[h] + log2f(l)) * 0.69314718055994531f : -INFINITY;
            const int hq = g * G + h;
            if (nch == 1) {
                __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)b * Hq + hq) * D;
                uint2 u;
                u.x = pack_bf16x2(o[h][0] * inv, o[h][1] * inv);
                u.y = pack_bf16x2(o[h][2] * inv, o[h][3] * inv);
                *reinterpret_cast<uint2*>(op + lane * 4) = u;
                if (lane == 0 && p.lse) p.lse[(size_t)b * Hq + hq] = lse_v;
            } else {
                float* op = p.part_o + ((size_t)f * Hq + hq) * D;
                *reinterpret_cast<float4*>(op + lane * 4) =
                    make_float4(o[h][0] * inv, o[h][1] * inv, o[h][2] * inv, o[h][3] * inv);
                if (lane == 0) p.part_lse[(size_t)f * Hq + hq] = lse_v;
            }
        }
    }
}

// One warp per (request, head) row whose request was split into several chunks.
__global__ void __launch_bounds__(256) merge_kernel(const Params p) {
    constexpr int D = HEAD_DIM;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int Hq = p.num_qo_heads;
    if (row >= (long long)p.batch * Hq) return;
    const int b = (int)(row / Hq), h = (int)(row % Hq);
    const int f0 = __ldg(p.chunk_off + b);
    const int nch = __ldg(p.chunk_off + b + 1) - f0;
    if (nch <= 1) return;
    float mx = -INFINITY;
    for (int c = lane; c < nch; c += 32) mx = fmaxf(mx, p.part_lse[(size_t)(f0 + c) * Hq + h]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int c = 0; c < nch; ++c) {
            const float w = __expf(p.part_lse[(size_t)(f0 + c) * Hq + h] - mx);
            const float4 v = *reinterpret_cast<const float4*>(
                p.part_o + ((size_t)(f0 + c) * Hq + h) * D + lane * 4);
            wsum += w;
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)b * Hq + h) * D;
    uint2 u;
    u.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    u.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(op + lane * 4) = u;
    if (lane == 0 && p.lse) p.lse[(size_t)b * Hq + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// ------------------------------------------------------------------ host launchers
cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream) {
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(pp);
    return cudaGetLastError();
}

template <int G>
static cudaError_t launch_decode_g(const Params& p, int num_sms, cudaStream_t stream) {
    static int blocks_per_sm[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (blocks_per_sm[dev] == 0) {
        int n = 0;
        cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<G>, WARPS * 32, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev] = n > 0 ? n : 1;
    }
    const int grid = num_sms * blocks_per_sm[dev];
    decode_kernel<G><<<grid, WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

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
    const long long rows = (long long)p.batch * p.num_qo_heads;
    const int grid = (int)((rows + 7) / 8);
    if (grid > 0) merge_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace decode
}  // namespace pgqa
