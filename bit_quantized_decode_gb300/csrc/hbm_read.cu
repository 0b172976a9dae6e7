// Pure-read bandwidth probe (w4_hbm_read): the read-only roofline bound of a
// weight-streaming decode.  "在香橙派上跑 Gemma4", §4.1 takes the device's
// measured pure read bandwidth (not a read+write copy) as the bound of the
// decode; this measures it on this device with the streaming machinery of the
// GEMVs: one block of eight warps per SM, each warp a ring of 4 KB slots fed
// by 1-D bulk copies (evict-first), bounded mbarrier waits.  Every 32-bit
// word read is folded into an XOR, written to *sink, so no read is dead.
#include "internal.h"
#include "ptx.cuh"

namespace w4k {

namespace {

constexpr int kReadWarps = 8;
constexpr int kReadThreads = kReadWarps * 32;
constexpr int kReadSlot = 4096;       // bytes per ring slot (one bulk copy)
constexpr int kReadStages = 6;        // slots per warp
constexpr uint64_t kReadTimeoutNs = 250ull * 1000ull * 1000ull;

// Block b reads the contiguous range [b0, b1) of 4 KB chunks (the last chunk
// of the buffer may be shorter); warp w of the block takes chunks b0 + w,
// b0 + w + 8, ...
__global__ void __launch_bounds__(kReadThreads, 1) hbm_read_kernel(const uint8_t* __restrict__ buf,
                                                                   unsigned long long bytes, unsigned* sink,
                                                                   unsigned* err)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint8_t* ring = smem + 128 * ((kReadWarps * kReadStages * 8 + 127) / 128);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long nchunks = (bytes + kReadSlot - 1) / kReadSlot;
    const unsigned long long per = nchunks / gridDim.x;
    const unsigned long long rem = nchunks % gridDim.x;
    const unsigned long long b = blockIdx.x;
    const unsigned long long b0 = b * per + (b < rem ? b : rem);
    const unsigned long long b1 = b0 + per + (b < rem ? 1 : 0);

    uint8_t* my_ring = ring + static_cast<size_t>(warp) * kReadStages * kReadSlot;
    const uint32_t my_bars = smem_u32(bars + warp * kReadStages);
    if (lane == 0) {
        for (int s = 0; s < kReadStages; ++s) mbar_init(my_bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();

    unsigned long long next = b0 + warp;      // next chunk to issue
    int issued = 0, observed = 0;
    auto issue = [&](int slot) {
        if (lane == 0) {
            const unsigned long long off = next * kReadSlot;
            const uint32_t n = static_cast<uint32_t>(bytes - off < kReadSlot ? bytes - off : kReadSlot);
            if (issued >= kReadStages) fence_proxy_async_smem();
            mbar_arrive_expect_tx(my_bars + 8 * slot, n);
            bulk_g2s(smem_u32(my_ring + static_cast<size_t>(slot) * kReadSlot), buf + off, n, my_bars + 8 * slot,
                     pol);
        }
        next += kReadWarps;
        ++issued;
    };
#pragma unroll 1
    for (int s = 0; s < kReadStages && next < b1; ++s) issue(s);

    uint32_t acc = 0;
    bool dead = false;
    int slot = 0;
    uint32_t phase = 0;
    unsigned long long cur = b0 + warp;
#pragma unroll 1
    while (cur < b1 && !dead) {
        const bool ok = mbar_wait_bounded(my_bars + 8 * slot, phase, kReadTimeoutNs);
        if (!__all_sync(0xffffffffu, ok)) {
            dead = true;
            if (lane == 0 && err != nullptr) atomicExch(err, 0x52454144u);   // "READ"
            break;
        }
        ++observed;
        const unsigned long long off = cur * kReadSlot;
        const int n16 = static_cast<int>((bytes - off < kReadSlot ? bytes - off : kReadSlot) / 16);
        const uint4* src = reinterpret_cast<const uint4*>(my_ring + static_cast<size_t>(slot) * kReadSlot);
#pragma unroll 4
        for (int i = lane; i < n16; i += 32) {
            const uint4 v = src[i];
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        __syncwarp();
        if (next < b1) issue(slot);
        cur += kReadWarps;
        if (++slot == kReadStages) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // after a timeout: wait (bounded) for this warp's copies still in flight
    if (dead) {
        for (int k = observed; k < issued; ++k)
            if (!mbar_wait_bounded(my_bars + 8 * (k % kReadStages), static_cast<uint32_t>(k / kReadStages) & 1u,
                                   kReadTimeoutNs))
                break;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0 && acc != 0u) atomicXor(sink, acc);
}

}  // namespace

size_t hbm_read_smem() { return 128 * ((kReadWarps * kReadStages * 8 + 127) / 128) + kReadWarps * kReadStages * kReadSlot; }

cudaError_t launch_hbm_read(const void* buf, unsigned long long bytes, unsigned* sink, unsigned* err, int sms,
                            cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(sink, 0, sizeof(unsigned), s);
    if (e != cudaSuccess || bytes == 0) return e;
    static SmemLimit limit;
    const size_t smem = hbm_read_smem();
    e = raise_smem_limit(reinterpret_cast<const void*>(hbm_read_kernel), limit, smem);
    if (e != cudaSuccess) return e;
    const unsigned long long nchunks = (bytes + kReadSlot - 1) / kReadSlot;
    const unsigned grid = static_cast<unsigned>(nchunks < static_cast<unsigned long long>(sms) ? nchunks : sms);
    hbm_read_kernel<<<grid, kReadThreads, smem, s>>>(static_cast<const uint8_t*>(buf), bytes, sink, err);
    return cudaGetLastError();
}

// ------------------------------------------------- the timeout path, tested
// A wait that nothing completes: thread 0 of block 0 waits (bounded) for phase
// 0 of an mbarrier on which no thread arrives, and records the timeout in the
// device error word as every kernel's bounded waits do.  With `cluster`, two
// blocks form a cluster and block 0 waits with cluster-scope acquire (the
// K-split leader's wait) while block 1 leaves, as the other splits do.  The
// kernel always ends after `timeout_ns`: the error path of the waits runs on
// the GPU without a fault, and the context stays usable.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int cluster, unsigned long long timeout_ns, unsigned* err)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (cluster) cluster_sync();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const bool ok = cluster ? mbar_wait_cluster_bounded(b, 0u, timeout_ns) : mbar_wait_bounded(b, 0u, timeout_ns);
        if (!ok && err != nullptr) atomicExch(err, kErrWaitTimeout);
    }
    __syncwarp();
}

cudaError_t launch_wait_selftest(int cluster, unsigned long long timeout_ns, unsigned* err, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster ? 2u : 1u);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (cluster) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, wait_selftest_kernel, cluster, timeout_ns, err);
}

}  // namespace w4k
