// dequant.cu -- the pages of an FP8 E4M3 KV cache that a paged prefill reads, converted to
// K in bf16 and V in f16, for sm_103a.
//
// A paged prefill over an E4M3 cache whose requests have more query rows than the
// tensor-core E4M3 decode takes (16 / G) runs the prefill kernels' converted-page
// instances: their K/V tiles stream by TMA straight into the tensor cores' swizzled operand
// layout, which has no room for a conversion stage.  So the pages the call reads are
// converted first, into a pool in the workspace.  Both conversions are exact (every E4M3
// value is a bf16 and an f16 value).  K is bf16 because Q.K^T pairs it with the bf16
// queries; V is f16 so that P.V can take P rounded to f16 (11 bits) rather than bf16
// (8 bits).  The scales are not applied here: k_scale joins the score scale and v_scale
// the output scale of the prefill, as for the decode.  The extra traffic (one read of the
// E4M3 pages, one write and read of the 2-byte pool) is small next to a long prefill's
// tensor work.
// Sources: FlashInfer documentation, flashinfer_benchmark.py "Attention Flags"
// (--kv_dtype fp8_e4m3 for the prefill routines); FlashInfer documentation,
// flashinfer.prefill (BatchPrefillWithPagedKVCacheWrapper: the paged prefill itself).
//
// Two pool mappings, whichever pool is smaller:
//  * by page: the pool has the caller's num_pages pages and page p holds page p, so the
//    caller's page table is used as it is (a page shared by two requests is converted
//    twice, to the same bits);
//  * by table slot: the pool has batch x page_table_stride pages, page b * stride + j holds
//    the page of slot j of request b, and the kernel writes a table pointing there.
// Only the slots below ceil(kv_len / page_size) of each request are converted.  A kv_len
// outside 0..stride * page_size converts nothing (the prefill's plan reports it); a page
// id outside 0..num_pages-1 is reported as PGQA_DEV_BOUNDS and not read.
//
// The conversion runs beside the prefill's plan: the plan (one CTA) starts first and lets
// this grid launch at once; each CTA of this grid waits for the plan to complete before
// it exits, so that the attention kernel, which waits for this grid, sees the plan's work
// list as well as the pool.  Launched that way, the grid starts before the kernel ahead of
// it has ended, so it reads global memory through L2 (ld.global.cg) only.
#include "ptx.cuh"

namespace pgqa {
namespace dequant {

constexpr int THREADS = 256;

// 16 E4M3 bytes -> 16 f16 (exact: f16 holds every E4M3 value)
__device__ __forceinline__ void e4m3x16_to_f16(const uint4& raw, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(out[2 * i]), "=r"(out[2 * i + 1])
            : "r"(w[i]));
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// 16 E4M3 bytes -> 16 bf16, exactly (through f16, which holds every E4M3 value)
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4& raw, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h01, h23;
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(h01), "=r"(h23)
            : "r"(w[i]));
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        out[2 * i] = pack_bf16x2(f01.x, f01.y);
        out[2 * i + 1] = pack_bf16x2(f23.x, f23.y);
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// One CTA per table slot (grid-stride): the slot's page, K and V, 16 bytes per thread step.
__global__ void __launch_bounds__(THREADS) dequant_pages_kernel(const Params p) {
    const long long slots = (long long)p.batch * p.page_table_stride;
    const int units_per_slot = p.num_kv_heads * p.head_dim / 16;  // 16-byte units of one slot
    const int units = p.page_size * units_per_slot;
    for (long long sl = blockIdx.x; sl < slots; sl += gridDim.x) {
        const int b = (int)(sl / p.page_table_stride);
        const int j = (int)(sl % p.page_table_stride);
        if (p.table_out != nullptr && threadIdx.x == 0) p.table_out[sl] = (int)sl;
        int kv = __ldcg(p.kv_lens + b);
        if (kv < 0 || (long long)kv > (long long)p.page_table_stride * p.page_size) kv = 0;
        if ((long long)j * p.page_size >= kv) continue;  // uniform per CTA
        const int pid = __ldcg(p.page_table + sl);
        if (pid < 0 || pid >= p.num_pages) {
            if (threadIdx.x == 0) atomicOr(p.status, PGQA_DEV_BOUNDS);
            continue;
        }
        const long long dst_page = p.table_out != nullptr ? sl : pid;
        const uint8_t* ks = p.k8 + (long long)pid * p.page_stride;
        const uint8_t* vs = p.v8 + (long long)pid * p.page_stride;
        __nv_bfloat16* kd = static_cast<__nv_bfloat16*>(p.k16) + dst_page * (long long)units * 16;
        __nv_bfloat16* vd = static_cast<__nv_bfloat16*>(p.v16) + dst_page * (long long)units * 16;
        for (int u = threadIdx.x; u < units; u += THREADS) {
            const int slot = u / units_per_slot, r = u % units_per_slot;
            const int h = r / (p.head_dim / 16), c = r % (p.head_dim / 16);
            const long long src =
                (long long)slot * p.slot_stride + (long long)h * p.head_stride + c * 16;
            const uint4 rk = __ldcg(reinterpret_cast<const uint4*>(ks + src));
            const uint4 rv = __ldcg(reinterpret_cast<const uint4*>(vs + src));
            uint4 lo, hi;
            e4m3x16_to_bf16(rk, lo, hi);
            reinterpret_cast<uint4*>(kd + (long long)u * 16)[0] = lo;
            reinterpret_cast<uint4*>(kd + (long long)u * 16)[1] = hi;
            e4m3x16_to_f16(rv, lo, hi);  // V in f16: P.V then keeps P to f16 precision
            reinterpret_cast<uint4*>(vd + (long long)u * 16)[0] = lo;
            reinterpret_cast<uint4*>(vd + (long long)u * 16)[1] = hi;
        }
    }
    // the plan launched before this grid has completed, and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t launch_dequant(const Params& p, int num_sms, cudaStream_t stream) {
    const long long slots = (long long)p.batch * p.page_table_stride;
    if (slots <= 0) return cudaSuccess;
    const long long grid = slots < (long long)num_sms * 16 ? slots : (long long)num_sms * 16;
    // programmatic dependent launch: the grid may start while the plan still runs
    return launch_dependent(dequant_pages_kernel, (unsigned)grid, THREADS, 0, stream, p);
}

}  // namespace dequant
}  // namespace pgqa
