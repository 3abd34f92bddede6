// noalloc.cu -- purlin_all_reduce_noalloc: the staged (SNAC) AllReduce, with
// the reduced chunk staged, for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework that has reserved the
// GPU's memory for its own pool allocator (a direct cudaMalloc would fail, or
// would bypass the framework's accounting), a plugin that is forbidden to own
// device memory, or a latency-critical path that cannot afford the device-wide
// synchronization cudaMalloc/cudaFree may imply.  For them this file keeps the
// scratch memory the staged kernel needs -- its staging ring, its ready/free
// flags and a status word -- in ONE file-scope __device__ array of fixed size,
// created when the library is loaded and held by every GPU that loads it until
// the process exits.  The paper has no counterpart to this entry point.
//
// The array's name in host code is only a host-side stand-in, not a device
// address, so the device address is looked up with cudaGetSymbolAddress once
// per device (with that device current) and passed to the kernel.
#include "purlin.h"

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "plan.h"
#include "snac.h"

namespace purlin {
namespace {

constexpr size_t kScratchBytes = PURLIN_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusOffset = 0;               // one int, padded to 256 bytes
constexpr size_t kFlagsOffset = 256;
constexpr size_t kFlagWords = (64 * 1024 - 256) / 8;  // the rest of the header: 8160 flags
constexpr size_t kStagingOffset = 64 * 1024;      // the rest is the staging ring
constexpr size_t kStagingBytes = kScratchBytes - kStagingOffset;
constexpr size_t kDefaultChunk = 8 * 1024;  // 508 channels of 64-thread role CTAs
constexpr int kDefaultDepth = 2;
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kMaxDevices = 64;

static_assert(kFlagsOffset + kFlagWords * sizeof(uint64_t) <= kStagingOffset, "layout");

// Zero at load time; the flags hold epoch tags, so they never need clearing.
static __device__ __align__(256) char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
    std::mutex lock;
    bool ready = false;     // set once a lookup has succeeded; a failed one is retried
    char* base = nullptr;   // device address of g_noalloc_scratch on this device
    int sms = 0;
};

DeviceScratch g_devices[kMaxDevices];

// Look up the array's device address on the current device, once it succeeds.
// A failure (e.g. a first call made while a stream is being captured, where
// the lookup may be refused) is not remembered: the next call tries again.
bool set_up(DeviceScratch& d, int device)
{
    std::lock_guard<std::mutex> g(d.lock);
    if (d.ready) return true;
    void* ptr = nullptr;
    int sms = 0;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        (void)cudaGetLastError();   // do not leave the failure for the caller's next check
        return false;
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    d.base = static_cast<char*>(ptr);
    d.sms = sms;
    d.ready = true;
    return true;
}

bool overlaps(uint64_t a, uint64_t alen, uint64_t b, uint64_t blen)
{
    return alen && blen && a < b + blen && b < a + alen;
}

}  // namespace
}  // namespace purlin

using namespace purlin;

extern "C" PURLIN_API purlin_status_t purlin_all_reduce_noalloc(
    const void* const in[], void* const out[], int R, size_t count, purlin_dtype_t dtype,
    size_t chunk_bytes, int depth, int* device_status, purlin_stream_t stream)
{
    if (!in || !out || R < 1 || R > PURLIN_MAX_RANKS) return PURLIN_ERR_INVALID_ARG;
    if (dtype != PURLIN_F32 && dtype != PURLIN_BF16 && dtype != PURLIN_F16)
        return PURLIN_ERR_INVALID_ARG;
    if (depth < 0 || depth > 8 || chunk_bytes % 256) return PURLIN_ERR_INVALID_ARG;
    const size_t chunk = chunk_bytes ? chunk_bytes : kDefaultChunk;
    const int dep = depth ? depth : kDefaultDepth;
    // One channel's ring -- depth slots of one reduced chunk each -- must fit in
    // the static staging area.
    if (chunk > kStagingBytes / (size_t)dep) return PURLIN_ERR_INVALID_ARG;
    const size_t esz = dtype == PURLIN_F32 ? 4 : 2;
    if (count > UINT64_MAX / esz) return PURLIN_ERR_INVALID_ARG;
    const uint64_t bytes = (uint64_t)count * esz;
    uint64_t inp[kMaxRanks], outp[kMaxRanks];
    for (int r = 0; r < R; ++r) {
        inp[r] = reinterpret_cast<uint64_t>(in[r]);
        outp[r] = reinterpret_cast<uint64_t>(out[r]);
        if (bytes && (!inp[r] || !outp[r] || inp[r] % esz || outp[r] % esz))
            return PURLIN_ERR_INVALID_ARG;
    }
    for (int a = 0; a < R; ++a)
        for (int b = 0; b < R; ++b) {
            if (b > a && overlaps(outp[a], bytes, outp[b], bytes)) return PURLIN_ERR_INVALID_ARG;
            if (overlaps(inp[a], bytes, outp[b], bytes) && !(a == b && inp[a] == outp[b]))
                return PURLIN_ERR_INVALID_ARG;   // only out[r] == in[r] may alias
        }

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PURLIN_ERR_CUDA;
    if (device < 0 || device >= kMaxDevices) return PURLIN_ERR_UNSUPPORTED;
    DeviceScratch& d = g_devices[device];
    if (!set_up(d, device)) return PURLIN_ERR_CUDA;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int* status = device_status ? device_status
                                : reinterpret_cast<int*>(d.base + kStatusOffset);
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return PURLIN_ERR_CUDA;
    if (bytes == 0) return PURLIN_OK;

    Piece piece{0, 0, bytes, kEveryRank, kEveryRank};
    SnacRequest rq{};
    rq.coll = Coll::AllReduce;
    rq.R = R;
    rq.dtype = (int)dtype;
    rq.order = PURLIN_ORDER_FIXED;
    rq.esz = esz;
    rq.pieces = &piece;
    rq.npieces = 1;
#if defined(PURLIN_CHECKED)
    uint64_t ext[kMaxRanks];
    for (int r = 0; r < R; ++r) ext[r] = bytes;
    const CheckRanges check = call_ranges(
        R, inp, outp, ext, ext, violation_word(reinterpret_cast<int*>(d.base + kStatusOffset)));
    rq.check = &check;
#endif
    // The producers reduce the R inputs and stage the reduced chunk, the
    // consumers copy it to the R outputs: a slot holds one part, so the 8 MiB
    // array fits R + 1 times the channels that staging the R inputs would.
    rq.stage_y = true;
    for (int r = 0; r < R; ++r) { rq.in[r] = inp[r]; rq.out[r] = outp[r]; }
    SnacConfig cfg{};
    cfg.staging = d.base + kStagingOffset;
    cfg.staging_bytes = kStagingBytes;
    cfg.flags = reinterpret_cast<uint64_t*>(d.base + kFlagsOffset);
    cfg.flag_words = kFlagWords;
    cfg.status = status;
    cfg.chunk_bytes = chunk;
    cfg.depth = dep;
    cfg.channels = 0;
    cfg.sms = d.sms;
    cfg.timeout_ns = kTimeoutNs;
    cfg.inject_skip_notify = 0;
    SnacLaunch launch{};
    return snac_run_on_stack(rq, cfg, s, &launch);
}
