// LSE merge of partial attention results over KV blocks (Context Parallelism
// for Scalable Million-Token Inference, Appendix B, Eq. 4), and the device
// watchdog self-test.
//
// Memory-bound: every (row, head) unit reads n_parts LSE values and n_parts
// O rows and writes one O row.  d/8 threads share a unit, each owning 8
// consecutive channels (16-byte bf16 / 32-byte fp32 vector accesses), so a
// warp touches contiguous memory.
#include <cmath>

#include <cuda_bf16.h>

#include "ca_sm100.cuh"

namespace ca {
namespace {

struct MergeParams {
    const void *o[kMaxMergeParts];
    const float *lse[kMaxMergeParts];
    int32_t n;
    int32_t d;
    int64_t units;  // rows * heads
    void *out;
    float *lse_out;
};

template <bool IN_F32>
__device__ __forceinline__ void load8(const void *base, int64_t elem, float (&x)[8]) {
    if (IN_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + elem);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(base) + elem));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <bool IN_F32, bool OUT_F32>
__global__ void __launch_bounds__(256) ca_merge_kernel(const MergeParams p) {
    const int32_t tpu = p.d / 8;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t unit = gtid / tpu;
    const int32_t part = static_cast<int32_t>(gtid % tpu);
    if (unit >= p.units) return;
    float M = -INFINITY;
    for (int32_t s = 0; s < p.n; ++s) M = fmaxf(M, __ldg(p.lse[s] + unit));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    const int64_t elem = unit * p.d + part * 8;
    if (M != -INFINITY) {
        for (int32_t s = 0; s < p.n; ++s) {
            const float w = expf(__ldg(p.lse[s] + unit) - M);  // 0 for an empty part
            wsum += w;
            float x[8];
            load8<IN_F32>(p.o[s], elem, x);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, x[i], acc[i]);
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] *= inv;
    }
    if (OUT_F32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + elem);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
        uint4 w;
        w.x = dev::pack_bf16(acc[0], acc[1]);
        w.y = dev::pack_bf16(acc[2], acc[3]);
        w.z = dev::pack_bf16(acc[4], acc[5]);
        w.w = dev::pack_bf16(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + elem) = w;
    }
    if (part == 0 && p.lse_out) p.lse_out[unit] = (M == -INFINITY) ? -INFINITY : M + logf(wsum);
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait runs
// out, records kErrTimeout and returns.
__global__ void ca_watchdog_kernel(const DevCtl ctl) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        dev::mbar_init(&bar, 1);
        abort_flag = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const dev::Watchdog wd{&ctl, &abort_flag};
        dev::mbar_wait(&bar, 0, wd);
    }
}

}  // namespace

cudaError_t launch_merge(int32_t n_parts, const void *const *o_parts, const float *const *lse_parts,
                         int32_t parts_dtype, int64_t rows, int32_t heads, int32_t head_dim, void *o_out,
                         int32_t out_dtype, float *lse_out, cudaStream_t stream) {
    MergeParams p{};
    for (int32_t s = 0; s < n_parts; ++s) {
        p.o[s] = o_parts[s];
        p.lse[s] = lse_parts[s];
    }
    p.n = n_parts;
    p.d = head_dim;
    p.units = rows * heads;
    p.out = o_out;
    p.lse_out = lse_out;
    const int64_t threads = p.units * (head_dim / 8);
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const bool fi = parts_dtype == CA_DTYPE_FP32, fo = out_dtype == CA_DTYPE_FP32;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (fi && fo) ca_merge_kernel<true, true><<<grid, 256, 0, stream>>>(p);
    else if (fi) ca_merge_kernel<true, false><<<grid, 256, 0, stream>>>(p);
    else if (fo) ca_merge_kernel<false, true><<<grid, 256, 0, stream>>>(p);
    else ca_merge_kernel<false, false><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(const ca_plan *pl, int64_t limit_ns, cudaStream_t stream) {
    DevCtl ctl;
    ctl.err = pl->d_err;
    ctl.wait_limit_ns = static_cast<unsigned long long>(limit_ns);
    ca_watchdog_kernel<<<1, 32, 0, stream>>>(ctl);
    return cudaGetLastError();
}

}  // namespace ca
