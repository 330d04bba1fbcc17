// kq_probe.cu -- measurement aid: the throughput ceiling of the legacy warp-level int8 tensor path.
//
// The metric is quoted in int8 TOPS, and the int8 MMA available to sm_103a code is the warp-level
// mma.sync m16n8k32 s8 x s8 -> s32 (tcgen05 has no integer kind here).  This kernel saturates it:
// every warp issues independent MMAs on register operands (no memory traffic), four accumulator
// sets deep so that consecutive MMAs do not wait on one another.  The caller times the launch; the
// op count is returned on the host.  Nothing on the hot path uses it.
#include "kq_internal.cuh"

namespace kq {

constexpr int kProbeWarps = 8;   // warps per block
constexpr int kProbeChains = 4;  // independent accumulator sets per warp

__global__ void __launch_bounds__(kProbeWarps * 32) int8_mma_sync_probe_kernel(int64_t iters, int32_t *sink) {
    const int lane = threadIdx.x & 31;
    // operands that vary by lane so nothing is constant-folded
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * (uint32_t)((lane + i) & 7);
    b[0] = 0x01010101u * (uint32_t)(lane & 3);
    b[1] = 0x01010101u * (uint32_t)((lane >> 2) & 3);
    int32_t c[kProbeChains][4];
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[k][i] = 0;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < kProbeChains; ++k)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    int32_t s = 0;
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) s += c[k][0] + c[k][1] + c[k][2] + c[k][3];
    if (s == 0x7fffffff) *sink = s;  // practically never taken; keeps the MMAs live
}

}  // namespace kq

using namespace kq;

extern "C" kq_status kq_probe_int8_mma_sync(int64_t iters, int32_t *sink, double *ops, kq_stream_t stream) {
    if (iters <= 0 || !sink || !ops) return fail(KQ_ERR_INVALID_ARG, "kq_probe_int8_mma_sync: need iters > 0, sink, ops");
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(KQ_ERR_CUDA, "kq_probe_int8_mma_sync: no device");
    const unsigned blocks = (unsigned)sms * 4;  // 32 warps per SM
    int8_mma_sync_probe_kernel<<<blocks, kProbeWarps * 32, 0, (cudaStream_t)stream>>>(iters, sink);
    kq_status s = check_launch("kq_probe_int8_mma_sync");
    if (s != KQ_OK) return s;
    *ops = (double)blocks * kProbeWarps * (double)iters * kProbeChains * (2.0 * 16 * 8 * 32);
    return KQ_OK;
}
