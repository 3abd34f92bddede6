// zs_kernels.cu -- zero-staging ("ZS") Atom kernels for sm_103a.
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives",
// Figure 10: "Purlin-ZS omits staging" when buffers are directly accessible.  On
// one GPU every virtual rank's buffer is directly accessible, so the ZS kernels
// read the sources and write the destinations in one pass:
//   - zs_reduce: ReduceScatter(V) (one destination per segment) and the fused
//     AllReduce of Figure 6 (each summed unit written to all R outputs);
//   - zs_copy:   AllGather(V) (each unit written to all R outputs) and
//     AllToAll(V) (one destination per segment).
// Work is a flat space of tiles (plan.h) walked grid-stride by a resident grid;
// each CTA finds a tile's segment by binary search over the segments' first
// tiles, which sit in the kernel's constant parameter bank.
#include "atom.cuh"
#include "internal.h"

#include <mutex>
#include <unordered_map>

namespace purlin {

namespace {

template <int MAXSEG>
__device__ __forceinline__ const Segment& segment_of(const ZsParams<MAXSEG>& p, uint32_t t)
{
    int lo = 0, hi = (int)p.nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile0 <= t) lo = mid;
        else hi = mid - 1;
    }
    return p.seg[lo];
}

// Programmatic dependent launch: the grid may have been scheduled before the
// previous kernel on the stream finished; griddepcontrol.wait blocks until that
// kernel has completed and its writes are visible (it returns at once when the
// launch had no programmatic dependency).  Triggering dependents right after
// lets the next collective's CTAs be scheduled while this one runs.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ reduce

template <typename T, int ORDER, bool FAN_ALL, int BYTES>
__device__ __forceinline__ void reduce_vector(const ZsParams<kSegsSmall>& p, const Segment& s,
                                              uint64_t off, int R, uint64_t lpol, uint64_t spol)
{
    atom::Vec<BYTES> v[kMaxRanks];
    // All R loads are issued before the first add: R independent requests in
    // flight per thread.
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        if (r < R) atom::load(v[r], p.in[r] + s.src_off + off, lpol);
    atom::Vec<BYTES> o;
    atom::reduce_unit<T, ORDER, BYTES>(v, R, o);
    if (FAN_ALL) {
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) atom::store(p.out[r] + s.dst_off + off, o, spol);
    } else {
        atom::store(p.out[s.dst] + s.dst_off + off, o, spol);
    }
}

template <typename T, int ORDER, bool FAN_ALL>
__device__ __forceinline__ void reduce_element(const ZsParams<kSegsSmall>& p, const Segment& s,
                                               uint64_t off, int R)
{
    float v[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r) v[r] = (r < R) ? T::load1(p.in[r] + s.src_off + off) : 0.0f;
    float acc = atom::fold<ORDER>(v, R);
    if (FAN_ALL) {
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) T::store1(p.out[r] + s.dst_off + off, acc);
    } else {
        T::store1(p.out[s.dst] + s.dst_off + off, acc);
    }
}

template <typename T, int ORDER, bool FAN_ALL>
__global__ void __launch_bounds__(kThreads, 2)
zs_reduce_kernel(const __grid_constant__ ZsParams<kSegsSmall> p)
{
    pdl_enter();
    const int R = (int)p.R;
    const uint64_t lpol = atom::l2_policy(p.l2_load);
    const uint64_t spol = atom::l2_policy(p.l2_store);
    for (uint32_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const Segment& s = segment_of(p, t);
        const int ul = s.unit_log2;
        const uint64_t off = (uint64_t)(t - s.tile0) * tile_bytes(ul, kUnrollReduce) +
                             ((uint64_t)threadIdx.x << ul);
        if (off >= s.bytes) continue;
        if (ul == 5) reduce_vector<T, ORDER, FAN_ALL, 32>(p, s, off, R, lpol, spol);
        else if (ul == 4) reduce_vector<T, ORDER, FAN_ALL, 16>(p, s, off, R, lpol, spol);
        else reduce_element<T, ORDER, FAN_ALL>(p, s, off, R);
    }
}

// -------------------------------------------------------------------- copy

using atom::Unit;
using atom::load_unit;
using atom::store_unit;

template <int BYTES>
__device__ __forceinline__ void load_hinted(Unit<BYTES>& u, const char* p, uint64_t pol)
{
    if constexpr (BYTES >= 16) atom::load(u.v, p, pol);
    else load_unit<BYTES>(u, p);
}

template <int BYTES>
__device__ __forceinline__ void store_hinted(char* p, const Unit<BYTES>& u, uint64_t pol)
{
    if constexpr (BYTES >= 16) atom::store(p, u.v, pol);
    else store_unit<BYTES>(p, u);
}

// Atom::copy of one tile: kUnrollCopy units per thread, each warp access
// contiguous; every unit loaded once and stored to one or all R outputs.
template <int BYTES, bool FAN_ALL, int MAXSEG>
__device__ __forceinline__ void copy_tile(const ZsParams<MAXSEG>& p, const Segment& s,
                                          uint64_t base, uint64_t lpol, uint64_t spol)
{
    const uint64_t rem = s.bytes - base;
    const char* src = p.in[s.src] + s.src_off + base;
    Unit<BYTES> u[kUnrollCopy];
#pragma unroll
    for (int k = 0; k < kUnrollCopy; ++k) {
        const uint64_t o = (uint64_t)(k * kThreads + threadIdx.x) * BYTES;
        if (o < rem) load_hinted<BYTES>(u[k], src + o, lpol);
    }
#pragma unroll
    for (int k = 0; k < kUnrollCopy; ++k) {
        const uint64_t o = (uint64_t)(k * kThreads + threadIdx.x) * BYTES;
        if (o >= rem) continue;
        if (FAN_ALL) {
            for (int r = 0; r < (int)p.R; ++r) {
                char* dst = p.out[r] + s.dst_off + base + o;
                if (dst != src + o) store_hinted<BYTES>(dst, u[k], spol);  // in-place: skip
            }
        } else {
            store_hinted<BYTES>(p.out[s.dst] + s.dst_off + base + o, u[k], spol);
        }
    }
}

template <bool FAN_ALL, int MAXSEG>
__global__ void __launch_bounds__(kThreads, 2)
zs_copy_kernel(const __grid_constant__ ZsParams<MAXSEG> p)
{
    pdl_enter();
    const uint64_t lpol = atom::l2_policy(p.l2_load);
    const uint64_t spol = atom::l2_policy(p.l2_store);
    for (uint32_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const Segment& s = segment_of(p, t);
        const int ul = s.unit_log2;
        const uint64_t base = (uint64_t)(t - s.tile0) * tile_bytes(ul, kUnrollCopy);
        switch (ul) {
        case 5: copy_tile<32, FAN_ALL>(p, s, base, lpol, spol); break;
        case 4: copy_tile<16, FAN_ALL>(p, s, base, lpol, spol); break;
        case 3: copy_tile<8, FAN_ALL>(p, s, base, lpol, spol); break;
        case 2: copy_tile<4, FAN_ALL>(p, s, base, lpol, spol); break;
        case 1: copy_tile<2, FAN_ALL>(p, s, base, lpol, spol); break;
        default: copy_tile<1, FAN_ALL>(p, s, base, lpol, spol); break;
        }
    }
}

// ------------------------------------------------------------- dispatch

template <typename P>
cudaError_t launch(void (*kernel)(P), const P& params, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = params.pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, params);
}

using ReduceKernel = void (*)(ZsParams<kSegsSmall>);

template <typename T>
ReduceKernel pick_reduce(int order, bool fan_all)
{
    if (order == 0) return fan_all ? zs_reduce_kernel<T, 0, true> : zs_reduce_kernel<T, 0, false>;
    return fan_all ? zs_reduce_kernel<T, 1, true> : zs_reduce_kernel<T, 1, false>;
}

ReduceKernel reduce_kernel_for(int dtype, int order, bool fan_all)
{
    if (dtype == kF32) return pick_reduce<atom::F32>(order, fan_all);
    if (dtype == kBF16) return pick_reduce<atom::BF16>(order, fan_all);
    return pick_reduce<atom::F16>(order, fan_all);
}

// Resident CTAs per SM of a kernel at kThreads threads (cached per device).
int resident_ctas(const void* kernel)
{
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    uint64_t key = reinterpret_cast<uint64_t>(kernel) ^ ((uint64_t)dev << 56);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess || n < 1)
        n = 1;
    cache[key] = n;
    return n;
}

}  // namespace

cudaError_t zs_reduce_launch(const ZsParams<kSegsSmall>& p, int dtype, int order, bool fan_all,
                             int grid, cudaStream_t stream)
{
    return launch(reduce_kernel_for(dtype, order, fan_all), p, grid, stream);
}

int zs_reduce_resident_ctas(int dtype, int order, bool fan_all)
{
    return resident_ctas(reinterpret_cast<const void*>(reduce_kernel_for(dtype, order, fan_all)));
}

cudaError_t zs_copy_launch(const ZsParams<kSegsSmall>& p, bool fan_all, int grid,
                           cudaStream_t stream)
{
    return launch(fan_all ? zs_copy_kernel<true, kSegsSmall> : zs_copy_kernel<false, kSegsSmall>,
                  p, grid, stream);
}

cudaError_t zs_copy_launch(const ZsParams<kSegsLarge>& p, bool fan_all, int grid,
                           cudaStream_t stream)
{
    return launch(fan_all ? zs_copy_kernel<true, kSegsLarge> : zs_copy_kernel<false, kSegsLarge>,
                  p, grid, stream);
}

int zs_copy_resident_ctas(bool large, bool fan_all)
{
    const void* k;
    if (large)
        k = reinterpret_cast<const void*>(fan_all ? zs_copy_kernel<true, kSegsLarge>
                                                  : zs_copy_kernel<false, kSegsLarge>);
    else
        k = reinterpret_cast<const void*>(fan_all ? zs_copy_kernel<true, kSegsSmall>
                                                  : zs_copy_kernel<false, kSegsSmall>);
    return resident_ctas(k);
}

}  // namespace purlin
