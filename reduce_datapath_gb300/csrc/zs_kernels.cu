// zs_kernels.cu -- host-side selection and launch of the zero-staging Atom
// kernels (zs_kernels.cuh): which instantiation serves a call, its launch
// shape, its residency, and the one launch routine every planned call goes
// through (capi.cpp builds the parameter blocks).
#include "zs_kernels.cuh"

#include <mutex>

namespace purlin {
namespace {

// ------------------------------------------------------------- dispatch

using ReduceKernel = void (*)(ZsParams<kSegsSmall>);

// NR = kMaxRanks / units per thread.  The pairwise rank order keeps one unit
// per thread (NR = kMaxRanks).  SH: 0 no shifted segment, 1 shifted segments
// on one offset, 2 a sum whose ranks' sources sit on different offsets.
template <typename T, int THREADS, int NR, int SH>
ReduceKernel pick_reduce(int order, bool fan_all)
{
    if (order == 0)
        return fan_all ? zs_reduce_kernel<T, 0, true, THREADS, NR, SH>
                       : zs_reduce_kernel<T, 0, false, THREADS, NR, SH>;
    return fan_all ? zs_reduce_kernel<T, 1, true, THREADS, kMaxRanks, SH>
                   : zs_reduce_kernel<T, 1, false, THREADS, kMaxRanks, SH>;
}

template <int THREADS, int NR, int SH>
ReduceKernel reduce_kernel_t(int dtype, int order, bool fan_all)
{
    if (dtype == kF32) return pick_reduce<atom::F32, THREADS, NR, SH>(order, fan_all);
    if (dtype == kBF16) return pick_reduce<atom::BF16, THREADS, NR, SH>(order, fan_all);
    return pick_reduce<atom::F16, THREADS, NR, SH>(order, fan_all);
}

template <int SH>
ReduceKernel reduce_kernel_sh(int dtype, int order, bool fan_all, bool small, int unroll)
{
    if (small) return reduce_kernel_t<kSmallThreads, kMaxRanks, SH>(dtype, order, fan_all);
    switch (unroll) {
    case 4: return reduce_kernel_t<kThreads, kMaxRanks / 4, SH>(dtype, order, fan_all);
    case 2: return reduce_kernel_t<kThreads, kMaxRanks / 2, SH>(dtype, order, fan_all);
    default: return reduce_kernel_t<kThreads, kMaxRanks, SH>(dtype, order, fan_all);
    }
}

ReduceKernel reduce_kernel_for(int dtype, int order, bool fan_all, bool small, int unroll,
                               int shift_mode)
{
    if (shift_mode == 2) return reduce_kernel_sh<2>(dtype, order, fan_all, small, unroll);
    if (shift_mode == 1) return reduce_kernel_sh<1>(dtype, order, fan_all, small, unroll);
    return reduce_kernel_sh<0>(dtype, order, fan_all, small, unroll);
}

template <int MAXSEG, bool SH>
void (*copy_kernel_sh(bool fan_all, bool small))(ZsParams<MAXSEG>)
{
    if (small)
        return fan_all ? zs_copy_kernel<true, MAXSEG, kSmallThreads, 1, SH>
                       : zs_copy_kernel<false, MAXSEG, kSmallThreads, 1, SH>;
    return fan_all ? zs_copy_kernel<true, MAXSEG, kThreads, kUnrollCopy, SH>
                   : zs_copy_kernel<false, MAXSEG, kThreads, kUnrollCopy, SH>;
}

template <int MAXSEG>
const void* copy_kernel_for(bool fan_all, bool small, bool shifted)
{
    return shifted ? reinterpret_cast<const void*>(copy_kernel_sh<MAXSEG, true>(fan_all, small))
                   : reinterpret_cast<const void*>(copy_kernel_sh<MAXSEG, false>(fan_all, small));
}

const void* copy_kernel_any(bool large, bool fan_all, bool small, bool shifted)
{
    return large ? copy_kernel_for<kSegsLarge>(fan_all, small, shifted)
                 : copy_kernel_for<kSegsSmall>(fan_all, small, shifted);
}

// Resident CTAs per SM of a kernel at `threads` threads, cached per device in a
// fixed table (no heap allocation: the allocation-free AllReduce plans through
// this too).  At least 1.
int resident_ctas(const void* kernel, int threads)
{
    struct Entry { const void* kernel; int device; int threads; int n; };
    static std::mutex mu;
    static Entry cache[512];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kernel == kernel && cache[i].device == dev && cache[i].threads == threads)
            return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    if (used < 512) cache[used++] = Entry{kernel, dev, threads, n};
    return n;
}

constexpr int kBulkStages = 8;
constexpr size_t kBulkSmem = (size_t)kBulkStages * kBulkStageBytes;

// The bulk kernel's one-time shared-memory opt-in and residency, per device.
template <bool FAN_ALL, int MAXSEG>
cudaError_t bulk_setup(const void** func, int* resident_out)
{
    auto kernel = zs_copy_bulk_kernel<FAN_ALL, MAXSEG, kBulkStages>;
    static std::mutex mu;
    static bool ready[64] = {};
    static int resident[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kBulkSmem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kBulkThreads, kBulkSmem);
        if (e != cudaSuccess) return e;
        resident[dev] = n > 0 ? n : 1;
        ready[dev] = true;
    }
    if (func) *func = reinterpret_cast<const void*>(kernel);
    if (resident_out) *resident_out = resident[dev];
    return cudaSuccess;
}

cudaError_t bulk_setup_any(bool large, bool fan_all, const void** func, int* resident)
{
    if (large)
        return fan_all ? bulk_setup<true, kSegsLarge>(func, resident)
                       : bulk_setup<false, kSegsLarge>(func, resident);
    return fan_all ? bulk_setup<true, kSegsSmall>(func, resident)
                   : bulk_setup<false, kSegsSmall>(func, resident);
}

}  // namespace

int resident_ctas_of(const void* kernel, int threads)
{
    return resident_ctas(kernel, threads);
}

cudaError_t launch_kernel(const KernelLaunch& k, cudaStream_t stream)
{
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = k.pdl ? 1 : 0;
    ++n;
    if (k.cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(k.grid);
    cfg.blockDim = dim3(k.block);
    cfg.dynamicSmemBytes = k.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void* args[1] = {const_cast<unsigned char*>(k.params)};
    return cudaLaunchKernelExC(&cfg, k.func, args);
}

int reduce_unroll(int R, int order)
{
    if (order != 0) return 1;
    return R >= 5 ? 1 : R >= 3 ? 2 : 4;
}

void zs_reduce_select(KernelLaunch& k, int dtype, int order, bool fan_all, bool small, int R,
                      int shift_mode)
{
    k.func = reinterpret_cast<const void*>(
        reduce_kernel_for(dtype, order, fan_all, small, reduce_unroll(R, order), shift_mode));
    k.block = small ? kSmallThreads : kThreads;
    k.smem = 0;
    k.cooperative = false;
    k.params_bytes = sizeof(ZsParams<kSegsSmall>);
}

int zs_reduce_resident_ctas(int dtype, int order, bool fan_all, bool small, int R, int shift_mode)
{
    return resident_ctas(reinterpret_cast<const void*>(reduce_kernel_for(
                             dtype, order, fan_all, small, reduce_unroll(R, order), shift_mode)),
                         small ? kSmallThreads : kThreads);
}

void zs_copy_select(KernelLaunch& k, bool large, bool fan_all, bool small, bool shifted)
{
    k.func = copy_kernel_any(large, fan_all, small, shifted);
    k.block = small ? kSmallThreads : kThreads;
    k.smem = 0;
    k.cooperative = false;
    k.params_bytes = large ? sizeof(ZsParams<kSegsLarge>) : sizeof(ZsParams<kSegsSmall>);
}

int zs_copy_resident_ctas(bool large, bool fan_all, bool small, bool shifted)
{
    return resident_ctas(copy_kernel_any(large, fan_all, small, shifted),
                         small ? kSmallThreads : kThreads);
}

cudaError_t zs_copy_bulk_select(KernelLaunch& k, bool large, bool fan_all)
{
    cudaError_t e = bulk_setup_any(large, fan_all, &k.func, nullptr);
    k.block = kBulkThreads;
    k.smem = kBulkSmem;
    k.cooperative = false;
    k.params_bytes = large ? sizeof(ZsParams<kSegsLarge>) : sizeof(ZsParams<kSegsSmall>);
    return e;
}

int zs_copy_bulk_resident_ctas(bool large, bool fan_all)
{
    int n = 1;
    return bulk_setup_any(large, fan_all, nullptr, &n) == cudaSuccess ? n : 1;
}

static_assert(sizeof(ZsParams<kSegsLarge>) <= kMaxLaunchParams, "launch parameter block");

}  // namespace purlin
