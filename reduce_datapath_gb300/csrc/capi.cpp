// capi.cpp -- the C ABI (include/purlin.h): argument checks, handle, policy,
// and dispatch of each collective to the layout module and the Atom kernels.
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives":
// the layers of Figure 1 map onto this file as
//   collective naming (abstract, Figure 4)  -> the entry points below,
//   codesign policies (Figure 1)            -> choose_variant / grid sizing,
//   SNAC (abstract, Figure 6)               -> snac_kernels.cu,
//   Atom (abstract, Table 4)                -> atom.cuh, zs_kernels.cu.
#include "purlin.h"
#include "purlin_layout.h"
#include "purlin_debug.h"

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"
#include "plan.h"
#include "snac.h"

using namespace purlin;

// A zero-staging call whose large-message plan has fewer tiles than this runs
// one-warp CTAs.  Measured on GB300, R = 8, bf16, per launch in a CUDA graph
// (256-thread vs one-warp CTAs): AllReduce 1 MiB per rank (128 large tiles)
// 3.28 vs 3.02 us, 4 MiB (512) 8.05 vs 8.81 us; ReduceScatter 256 KiB (32)
// 1.93 vs 1.64 us, 1 MiB (128) 2.09 vs 2.32 us; AllGather 1 MiB out per rank
// (32) 5.42 vs 3.17 us, 4 MiB (128) 6.26 vs 6.37 us.
static long small_tiles_default(Coll coll) { return coll == Coll::AllReduce ? 256 : 64; }

struct purlin_handle {
    int R = 0;
    int device = 0;
    int sms = 0;
    size_t l2_bytes = 0;
    // SNAC staging ring, flags and the device status word (owned).
    size_t staging_bytes = 0;
    char* staging = nullptr;
    uint64_t* flags = nullptr;
    size_t flag_words = 0;
    int* status = nullptr;
    // policy (0 = automatic)
    size_t chunk_bytes = 0;
    int depth = 0;
    int ctas = 0;
    int variant = PURLIN_VARIANT_AUTO;
    int order = PURLIN_ORDER_FIXED;
    uint64_t timeout_ns = 1000000000ull;
    int max_unit_log2 = 0;   // 0: automatic (32 B; 16 B for small sums)
    int l2_load = -1;        // -1: per collective; else kL2Normal/EvictFirst/EvictLast
    int l2_store = -1;
    int l2_coll_load[4] = {-1, -1, -1, -1};   // per-collective overrides (by Coll)
    int l2_coll_store[4] = {-1, -1, -1, -1};
    bool pdl = true;         // programmatic dependent launch of zero-staging kernels
    long small_tiles = -1;   // below this many large tiles: one-warp CTAs (-1: per collective)
    int atom = PURLIN_ATOM_AUTO;
    int direction = PURLIN_DIRECTION_AUTO;
    int inject = 0;  // purlin_debug_inject, one staged call
    purlin_launch_info_t last{};
    // purlin_plan_begin .. purlin_plan_end: the call is planned, not launched
    bool recording = false;
    purlin_plan* recorded = nullptr;
};

// One planned collective call: a kernel launch with its parameter block, or the
// copy-engine copies of a kernel-less AllGather / AllToAll, or nothing (an
// empty call).
struct CopyOp {
    void* dst;
    const void* src;
    size_t bytes;
};

struct purlin_plan {
    purlin_handle_t h = nullptr;
    int device = 0;
    int kind = 0;  // 0 nothing, 1 kernel, 2 copies, 3 kernel k then kernel k2
    purlin::KernelLaunch k;
    purlin::KernelLaunch k2;
    std::vector<CopyOp> copies;
    purlin_launch_info_t info{};
};

namespace {

constexpr int kVersionMajor = 1;
constexpr int kVersionMinor = 0;
// Half the 129 MB L2: at R = 8 and the default chunks every kind fits a
// channel on every resident CTA pair (a 32 MiB ring held the inputs-staged
// ReduceScatter and the AllToAllV to 128 channels: 218.9 and 275.3 us at 64 MiB
// per rank against 186.9 and 253.9 us with 152 channels here).
constexpr size_t kDefaultStaging = 64ull << 20;
constexpr size_t kFlagWords = 8192;

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

size_t elem_bytes(int dtype)
{
    switch (dtype) {
    case kF32: return 4;
    case kBF16: return 2;
    case kF16: return 2;
    case kU8: return 1;
    default: return 0;
    }
}

bool overlaps(uint64_t a, uint64_t alen, uint64_t b, uint64_t blen)
{
    if (alen == 0 || blen == 0) return false;
    return a < b + blen && b < a + alen;
}

// Pointer, alignment and aliasing rules of purlin.h for one call.
purlin_status_t check_buffers(Coll coll, int R, const uint64_t* in, const uint64_t* out,
                              const uint64_t* in_ext, const uint64_t* out_ext, size_t esz,
                              bool reduce, const size_t* counts, const size_t* da)
{
    for (int r = 0; r < R; ++r) {
        if ((in_ext[r] && !in[r]) || (out_ext[r] && !out[r])) return PURLIN_ERR_INVALID_ARG;
        if (in[r] + in_ext[r] < in[r] || out[r] + out_ext[r] < out[r]) return PURLIN_ERR_INVALID_ARG;
        if (reduce && ((in_ext[r] && in[r] % esz) || (out_ext[r] && out[r] % esz)))
            return PURLIN_ERR_INVALID_ARG;
    }
    // Output blocks inside one buffer must not overlap each other.
    if (coll == Coll::AllGather) {
        for (int a = 0; a < R; ++a)
            for (int b = a + 1; b < R; ++b) {
                uint64_t sa = (da ? da[a] : 0), sb = (da ? da[b] : 0);
                if (!da) {
                    for (int m = 0; m < a; ++m) sa += counts[m];
                    for (int m = 0; m < b; ++m) sb += counts[m];
                }
                if (overlaps(sa, counts[a], sb, counts[b])) return PURLIN_ERR_INVALID_ARG;
            }
    }
    // Outputs are pairwise disjoint.
    for (int a = 0; a < R; ++a)
        for (int b = a + 1; b < R; ++b)
            if (overlaps(out[a], out_ext[a], out[b], out_ext[b])) return PURLIN_ERR_INVALID_ARG;
    // An output may meet an input only in the in-place forms of purlin.h.
    for (int r = 0; r < R; ++r)
        for (int j = 0; j < R; ++j) {
            if (!overlaps(in[r], in_ext[r], out[j], out_ext[j])) continue;
            bool allowed = false;
            if (r == j) {
                if (coll == Coll::AllReduce) {
                    allowed = in[r] == out[r];
                } else if (coll == Coll::ReduceScatter) {
                    uint64_t d = 0;
                    if (da) d = da[r];
                    else for (int m = 0; m < r; ++m) d += counts[m];
                    allowed = out[r] == in[r] + d * esz;
                } else if (coll == Coll::AllGather) {
                    uint64_t d = 0;
                    if (da) d = da[r];
                    else for (int m = 0; m < r; ++m) d += counts[m];
                    allowed = in[r] == out[r] + d * esz;
                }
            }
            if (!allowed) return PURLIN_ERR_INVALID_ARG;
        }
    return PURLIN_OK;
}

}  // namespace

void purlin::add_range(CheckRanges& c, uint64_t lo, uint64_t bytes)
{
    if (bytes == 0 || c.n >= (uint32_t)kMaxCheckRanges) return;
    c.lo[c.n] = lo;
    c.hi[c.n] = lo + bytes;
    ++c.n;
}

CheckRanges purlin::call_ranges(int R, const uint64_t* in, const uint64_t* out,
                                const uint64_t* in_ext, const uint64_t* out_ext,
                                unsigned long long* bad)
{
    CheckRanges c;
    std::memset(&c, 0, sizeof(c));
    c.bad = bad;
    for (int r = 0; r < R; ++r) {
        add_range(c, in[r], in_ext[r]);
        add_range(c, out[r], out_ext[r]);
    }
    return c;
}

namespace {

// Launch-wide knobs of the zero-staging kernels.
struct ZsKnobs {
    int tile_units;
    int max_unit_log2;
    bool allow_shift;   // shifted bodies (vector kernels; the TMA bulk Atom has none)
    uint32_t l2_load;
    uint32_t l2_store;
    bool pdl;
};

// Measured on GB300 (64 MiB per rank, R = 8, bf16):
//  - with the 16-wave grid every collective runs best with 32-byte units
//    (AllReduce 154.8 vs 157.1 us, ReduceScatter 90.1 vs 97.4 us); small sums
//    use 16-byte units (replan_small), which doubles their CTAs;
//  - every source is read exactly once, so loads are evict-first; outputs are
//    written evict-first except the ReduceScatter's, which a following
//    collective (the AllGather of a ReduceScatter -> AllGather pair) reads
//    next.  In that pair the AllGather's reads then hit L2 and DRAM sees
//    almost only its writes: AllGather 104.3 -> 90.2 us, ReduceScatter
//    108.8 -> 98.5 us, the pair 5599 -> 6332 GB/s.
// bulk: the plan is for the TMA bulk Atom (copies only).
ZsKnobs zs_knobs(const purlin_handle* h, Coll coll, bool bulk)
{
    ZsKnobs k;
    const bool reduce = coll == Coll::ReduceScatter || coll == Coll::AllReduce;
    bulk = bulk && !reduce;
    k.tile_units = reduce ? kThreads * reduce_unroll(h->R, h->order)
                          : (bulk ? kTileUnitsBulk : kTileUnitsCopy);
    k.max_unit_log2 = h->max_unit_log2 ? h->max_unit_log2 : 5;
    k.allow_shift = !bulk;
    k.l2_load = h->l2_load >= 0 ? (uint32_t)h->l2_load : kL2EvictFirst;
    k.l2_store = h->l2_store >= 0 ? (uint32_t)h->l2_store
                                  : (coll == Coll::ReduceScatter ? kL2Normal : kL2EvictFirst);
    const int ci = (int)coll;
    if (h->l2_coll_load[ci] >= 0) k.l2_load = (uint32_t)h->l2_coll_load[ci];
    if (h->l2_coll_store[ci] >= 0) k.l2_store = (uint32_t)h->l2_coll_store[ci];
    k.pdl = h->pdl;
    return k;
}

template <int MAXSEG>
purlin_status_t make_params(ZsParams<MAXSEG>& p, const Piece* pieces, int npieces, int R,
                            const uint64_t* in, const uint64_t* out, size_t esz, bool reduce,
                            const ZsKnobs& k, int* status, const CheckRanges& check)
{
    const int max_unit_log2 = k.max_unit_log2;
    std::memset(&p, 0, sizeof(p));
#if defined(PURLIN_CHECKED)
    p.check = check;
#else
    (void)check;
#endif
    p.l2_load = k.l2_load;
    p.l2_store = k.l2_store;
    p.pdl = k.pdl ? 1u : 0u;
    p.status = status;
    for (int r = 0; r < R; ++r) {
        p.in[r] = reinterpret_cast<const char*>(in[r]);
        p.out[r] = reinterpret_cast<char*>(out[r]);
    }
    p.R = (uint32_t)R;
    p.tile_units = (uint32_t)k.tile_units;
    uint32_t ntiles = 0;
    int n = layout_segments(pieces, npieces, R, in, out, esz, reduce, k.tile_units,
                            max_unit_log2, k.allow_shift, p.seg, MAXSEG, &ntiles);
    if (n < 0) return PURLIN_ERR_UNSUPPORTED;
    if (reduce && max_unit_log2 > 4) {
        // the kernels that serve shifted sums take 16-byte vector bodies only
        bool shifted = false;
        for (int i = 0; i < n; ++i) shifted |= p.seg[i].shift != 0;
        if (shifted)
            n = layout_segments(pieces, npieces, R, in, out, esz, reduce, k.tile_units, 4,
                                k.allow_shift, p.seg, MAXSEG, &ntiles);
        if (n < 0) return PURLIN_ERR_UNSUPPORTED;
    }
    p.nseg = (uint32_t)n;
    p.ntiles = ntiles;
    return PURLIN_OK;
}

// Which kernels a plan needs: 0 no shifted body, 1 shifted bodies whose
// sources share one offset, 2 a sum whose ranks' sources sit on different ones.
template <int MAXSEG>
int has_shift(const ZsParams<MAXSEG>& p)
{
    int mode = 0;
    for (uint32_t i = 0; i < p.nseg; ++i) {
        if (p.seg[i].shift & kShiftPerRank) return 2;
        if (p.seg[i].shift) mode = 1;
    }
    return mode;
}

// Small messages: when the large-message plan has fewer than h->small_tiles
// tiles (of kTileUnitsReduce units for sums, kTileUnitsCopy for copies), the call runs one-warp CTAs over one-warp tiles instead, so that its
// few KiB spread over many SMs rather than queue in the load/store path of a
// few.  Returns true (and the re-planned params) if so.
template <int MAXSEG>
bool replan_small(const purlin_handle* h, Coll coll, ZsParams<MAXSEG>& p, const Piece* pieces,
                  int npieces, int R, const uint64_t* in, const uint64_t* out, size_t esz,
                  bool reduce, ZsKnobs& k, const CheckRanges& check)
{
    const long threshold = h->small_tiles >= 0 ? h->small_tiles : small_tiles_default(coll);
    // counted in tiles of one unit per thread for sums, whatever reduce_unroll
    // gave, so that the switch sits at the same message size for every R
    const long scale = reduce ? std::max(1, (int)k.tile_units / kTileUnitsReduce) : 1;
    if ((long)p.ntiles * scale >= threshold) return false;
    ZsKnobs ks = k;
    ks.tile_units = kTileUnitsSmall;
    if (reduce && !h->max_unit_log2) ks.max_unit_log2 = std::min(ks.max_unit_log2, 4);
    // A small message cannot crowd other data out of L2, and a caller that
    // repeats it (or has just written its inputs) finds it there: no
    // evict-first marking, which would let any other resident data outlast it.
    const int ci = (int)coll;
    if (h->l2_load < 0 && h->l2_coll_load[ci] < 0) ks.l2_load = kL2Normal;
    if (h->l2_store < 0 && h->l2_coll_store[ci] < 0) ks.l2_store = kL2Normal;
    if (make_params(p, pieces, npieces, R, in, out, esz, reduce, ks, p.status, check) !=
        PURLIN_OK) {
        // cannot happen (same segments, more tiles of a smaller size fit in
        // 32 bits only if the large plan did); keep the large plan
        make_params(p, pieces, npieces, R, in, out, esz, reduce, k, p.status, check);
        return false;
    }
    k = ks;
    return true;
}

size_t algorithmic_bytes(Coll coll, int R, const size_t* counts, size_t count, size_t esz)
{
    uint64_t total = 0;
    switch (coll) {
    case Coll::ReduceScatter:
        for (int k = 0; k < R; ++k) total += counts[k];
        return (size_t)((uint64_t)(R + 1) * total * esz);
    case Coll::AllGather:
        for (int k = 0; k < R; ++k) total += counts[k];
        return (size_t)((uint64_t)(R + 1) * total * esz);
    case Coll::AllReduce:
        return (size_t)(2ull * R * count * esz);
    case Coll::AllToAllV:
        for (int i = 0; i < R * R; ++i) total += counts[i];
        return (size_t)(2ull * total * esz);
    }
    return 0;
}

// Zero-staging grid: by default 16 CTAs per resident CTA slot, each taking a
// few tiles (grid-stride), rather than one resident wave walking all of them.
// The block scheduler then hands the remaining CTAs to whichever SMs drain
// first, so SMs that see slower memory take less of the work instead of setting
// the time.  Measured on GB300, R = 8, bf16, 64 MiB per rank (one resident
// wave -> 16 waves): ReduceScatter 92.5 -> 90.5 us, AllGather 102.0 -> 93.7 us,
// AllReduce 171.3 -> 157.8 us, AllToAllV 173.7 -> 155.5 us; AllGather with
// 1 GiB out per rank 1634 -> 1460 us.  One CTA per tile is slower again
// (AllReduce 161.5 us): a CTA's launch costs about as much as a tile.
// The TMA bulk Atom (one resident CTA per SM, each setting up a shared-memory
// ring) is best at 4 waves: AllGather 96.2 us at 608 CTAs vs 100.3 at 2432.
constexpr long kGridWaves = 16;
constexpr long kGridWavesBulk = 4;

int zs_grid(const purlin_handle* h, uint32_t ntiles, int resident, long waves = kGridWaves)
{
    if (ntiles == 0) return 0;
    long g = h->ctas > 0 ? h->ctas : (long)h->sms * resident * waves;
    return (int)std::max<long>(1, std::min<long>(g, (long)ntiles));
}

// The AllGather's pieces by destination: one per (destination, source),
// destination by destination, in-place blocks dropped.  Returns their count.
int pull_pieces(const Piece* pieces, int np, int R, const uint64_t* in, const uint64_t* out,
                Piece* pulled)
{
    int n = 0;
    for (int j = 0; j < R; ++j)
        for (int i = 0; i < np; ++i) {
            Piece e = pieces[i];
            e.dst = (uint8_t)j;
            if (in[e.src] + e.src_off == out[j] + e.dst_off) continue;  // in place
            pulled[n++] = e;
        }
    return n;
}

// Whether the R output buffers share one 16-byte alignment.
bool outputs_share_grid(const uint64_t* out, int R)
{
    for (int r = 1; r < R; ++r)
        if ((out[r] ^ out[0]) & 15u) return false;
    return true;
}

// Whether a copy's plan on the vector kernels holds a shifted body.
bool needs_shift(const Piece* pieces, int np, int R, const uint64_t* in, const uint64_t* out,
                 size_t esz, const ZsKnobs& knobs)
{
    Segment segs[kSegsLarge];
    uint32_t ntiles = 0;
    const int n = layout_segments(pieces, np, R, in, out, esz, false, kTileUnitsCopy,
                                  knobs.max_unit_log2, true, segs, kSegsLarge, &ntiles);
    for (int i = 0; i < n; ++i)
        if (segs[i].shift) return true;
    return false;
}

bool wants_staged(const purlin_handle* h)
{
    return h->variant == PURLIN_VARIANT_STAGED || h->variant == PURLIN_VARIANT_STAGED_Y;
}

// One collective call as planned: its arguments after validation.
struct Call {
    purlin_handle_t h;
    Coll coll;
    int R;
    int dtype;
    size_t esz;
    bool reduce;
    const uint64_t* in;
    const uint64_t* out;
    const Piece* pieces;
    int np;
    const CheckRanges* check;  // the call's buffers (checked builds test against them)
    const uint64_t* in_ext;    // bytes read from each input
    const uint64_t* out_ext;   // bytes touched in each output
};

// What a call launches: nothing (kind 0), kernel k (1), copy-engine copies
// (2), or kernel k then kernel k2 (3), with the launch record.
struct Launches {
    KernelLaunch& k;
    KernelLaunch& k2;
    std::vector<CopyOp>& copies;
    purlin_launch_info_t& info;
    int kind = 0;
};

// SNAC: one cooperative launch of producer / consumer (/ gatherer) CTAs.
purlin_status_t plan_staged(const Call& c, Launches& L)
{
    purlin_handle_t h = c.h;
    SnacRequest rq{};
    rq.coll = c.coll;
    rq.R = c.R;
    rq.dtype = c.dtype;
    rq.order = h->order;
    rq.esz = c.esz;
    rq.pieces = c.pieces;
    rq.npieces = c.np;
    rq.stage_y = h->variant == PURLIN_VARIANT_STAGED_Y;
    for (int r = 0; r < c.R; ++r) { rq.in[r] = c.in[r]; rq.out[r] = c.out[r]; }
    SnacConfig cfg{};
    cfg.staging = h->staging;
    cfg.staging_bytes = h->staging_bytes;
    cfg.flags = h->flags;
    cfg.flag_words = h->flag_words;
    cfg.status = h->status;
    cfg.chunk_bytes = h->chunk_bytes;
    cfg.depth = h->depth;
    cfg.channels = h->ctas;
    cfg.sms = h->sms;
    cfg.timeout_ns = h->timeout_ns;
    cfg.inject_skip_notify = h->inject == 1;
#if defined(PURLIN_CHECKED)
    rq.check = c.check;
#endif
    SnacLaunch sl{};
    purlin_status_t st = snac_plan(rq, cfg, L.k, &sl);
    if (st != PURLIN_OK) return st;
    if (h->inject == 1) h->inject = 0;
    L.kind = L.k.grid > 0 ? 1 : 0;
    L.info.variant = h->variant;
    L.info.kernels = sl.kernels;
    L.info.grid = sl.grid;
    L.info.block = sl.block;
    L.info.depth = sl.depth;
    L.info.chunk_bytes = sl.chunk_bytes;
    return PURLIN_OK;
}

// No kernel: every block goes to every destination through the copy engines,
// one asynchronous copy each, in stream order.
void plan_copy_engine(const Call& c, Launches& L)
{
    for (int i = 0; i < c.np; ++i) {
        const Piece& pc = c.pieces[i];
        const char* src = reinterpret_cast<const char*>(c.in[pc.src]) + pc.src_off;
        for (int j = 0; j < c.R; ++j) {
            if (pc.dst != kEveryRank && pc.dst != j) continue;
            char* dst = reinterpret_cast<char*>(c.out[j]) + pc.dst_off;
            if (dst == src) continue;  // in-place AllGather block
            L.copies.push_back(CopyOp{dst, src, (size_t)pc.bytes});
        }
    }
    L.kind = L.copies.empty() ? 0 : 2;
    L.info.kernels = 0;
    L.info.grid = 0;
    L.info.block = 0;
    L.info.chunk_bytes = 0;
}

// Copies with one destination per piece: AllToAll(V), and AllGather by
// destination (pull, or outputs on different 16-byte alignments, which no one
// fan-out body can be aligned to; single-destination pieces can each take a
// shifted body where their source is off their output's grid).
purlin_status_t plan_by_destination(const Call& c, ZsKnobs knobs, bool bulk, Launches& L)
{
    purlin_handle_t h = c.h;
    ZsParams<kSegsLarge>& p = *reinterpret_cast<ZsParams<kSegsLarge>*>(L.k.params);
    const Piece* plan = c.pieces;
    int nplan = c.np;
    Piece pulled[kMaxRanks * kMaxRanks];
    if (c.coll == Coll::AllGather) {
        // one piece per (destination, source), destination by destination;
        // every source is read R times (from L2 after the first read, hence
        // normal priority for the loads)
        nplan = pull_pieces(c.pieces, c.np, c.R, c.in, c.out, pulled);
        plan = pulled;
        if (h->l2_load < 0 && h->l2_coll_load[(int)c.coll] < 0) knobs.l2_load = kL2Normal;
    }
    purlin_status_t st =
        make_params(p, plan, nplan, c.R, c.in, c.out, c.esz, false, knobs, h->status, *c.check);
    if (st != PURLIN_OK) return st;
    int grid;
    if (bulk) {
        grid = zs_grid(h, p.ntiles, zs_copy_bulk_resident_ctas(true, false), kGridWavesBulk);
        if (zs_copy_bulk_select(L.k, true, false) != cudaSuccess) return PURLIN_ERR_CUDA;
        L.info.block = kBulkThreads;
    } else {
        const bool small = replan_small(h, c.coll, p, plan, nplan, c.R, c.in, c.out, c.esz, false,
                                        knobs, *c.check);
        const bool sh = has_shift(p) != 0;
        grid = zs_grid(h, p.ntiles, zs_copy_resident_ctas(true, false, small, sh));
        zs_copy_select(L.k, true, false, small, sh);
        if (small) L.info.block = kSmallThreads;
    }
    L.k.grid = (unsigned)grid;
    L.k.pdl = p.pdl != 0;
    L.kind = grid > 0 ? 1 : 0;
    L.info.grid = grid;
    L.info.kernels = grid > 0;
    L.info.chunk_bytes = tile_bytes(knobs.max_unit_log2, knobs.tile_units);
    return PURLIN_OK;
}

// AllReduce into outputs on different 16-byte alignments: no fan-out body
// fits them all.  Sum into out[0] (one destination: a shifted body where the
// sources are off its grid), then copy out[0] to the other outputs
// (single-destination shifted copies): (2R + 1) / 2R of the fused traffic
// instead of element accesses.
purlin_status_t plan_all_reduce_split(const Call& c, const ZsKnobs& knobs, Launches& L)
{
    purlin_handle_t h = c.h;
    const int R = c.R;
    ZsParams<kSegsSmall>& p = *reinterpret_cast<ZsParams<kSegsSmall>*>(L.k.params);
    Piece sum = c.pieces[0];
    sum.dst = 0;
    ZsKnobs ks = knobs;
    if (h->l2_store < 0 && h->l2_coll_store[(int)c.coll] < 0) ks.l2_store = kL2Normal;
    purlin_status_t st =
        make_params(p, &sum, 1, R, c.in, c.out, c.esz, true, ks, h->status, *c.check);
    if (st != PURLIN_OK) return st;
    const bool small = replan_small(h, c.coll, p, &sum, 1, R, c.in, c.out, c.esz, true, ks,
                                    *c.check);
    const int sh = has_shift(p);
    const int grid =
        zs_grid(h, p.ntiles, zs_reduce_resident_ctas(c.dtype, h->order, false, small, R, sh));
    zs_reduce_select(L.k, c.dtype, h->order, false, small, R, sh);
    L.k.grid = (unsigned)grid;
    L.k.pdl = p.pdl != 0;

    ZsParams<kSegsSmall>& p2 = *reinterpret_cast<ZsParams<kSegsSmall>*>(L.k2.params);
    uint64_t from[kMaxRanks];
    Piece copies[kMaxRanks];
    int nc = 0;
    for (int r = 0; r < R; ++r) from[r] = c.out[0];
    for (int j = 1; j < R; ++j) {
        if (c.out[j] == c.out[0]) continue;
        copies[nc++] = Piece{sum.dst_off, sum.dst_off, sum.bytes, 0, (uint8_t)j};
    }
    ZsKnobs kc = zs_knobs(h, Coll::AllToAllV, false);  // vector copies
    st = make_params(p2, copies, nc, R, from, c.out, c.esz, false, kc, h->status, *c.check);
    if (st != PURLIN_OK) return st;
    const bool small2 = replan_small(h, Coll::AllToAllV, p2, copies, nc, R, from, c.out, c.esz,
                                     false, kc, *c.check);
    const bool sh2 = has_shift(p2) != 0;
    const int grid2 = zs_grid(h, p2.ntiles, zs_copy_resident_ctas(false, false, small2, sh2));
    zs_copy_select(L.k2, false, false, small2, sh2);
    L.k2.grid = (unsigned)grid2;
    L.k2.pdl = p2.pdl != 0;
    L.kind = grid > 0 ? (grid2 > 0 ? 3 : 1) : 0;
    L.info.grid = grid;
    L.info.kernels = (grid > 0) + (grid2 > 0);
    if (small) L.info.block = kSmallThreads;
    L.info.chunk_bytes = tile_bytes(ks.max_unit_log2, ks.tile_units);
    return PURLIN_OK;
}

// The zero-staging kernel of ReduceScatter(V), AllReduce (fused: each sum
// written to all R outputs) and AllGather(V) (push: each source tile written
// to all R outputs).
purlin_status_t plan_zs(const Call& c, const ZsKnobs& knobs, bool bulk, Launches& L)
{
    purlin_handle_t h = c.h;
    ZsKnobs kn = knobs;
    ZsParams<kSegsSmall>& p = *reinterpret_cast<ZsParams<kSegsSmall>*>(L.k.params);
    purlin_status_t st = make_params(p, c.pieces, c.np, c.R, c.in, c.out, c.esz, c.reduce, kn,
                                     h->status, *c.check);
    if (st != PURLIN_OK) return st;
    const bool fan_all = c.coll == Coll::AllGather || c.coll == Coll::AllReduce;
    int grid;
    if (bulk) {
        grid = zs_grid(h, p.ntiles, zs_copy_bulk_resident_ctas(false, fan_all), kGridWavesBulk);
        if (zs_copy_bulk_select(L.k, false, fan_all) != cudaSuccess) return PURLIN_ERR_CUDA;
        L.info.block = kBulkThreads;
    } else {
        const bool small = replan_small(h, c.coll, p, c.pieces, c.np, c.R, c.in, c.out, c.esz,
                                        c.reduce, kn, *c.check);
        if (c.reduce) {
            const int sh = has_shift(p);
            grid = zs_grid(h, p.ntiles,
                           zs_reduce_resident_ctas(c.dtype, h->order, fan_all, small, c.R, sh));
            zs_reduce_select(L.k, c.dtype, h->order, fan_all, small, c.R, sh);
        } else {
            const bool sh = has_shift(p) != 0;
            grid = zs_grid(h, p.ntiles, zs_copy_resident_ctas(false, fan_all, small, sh));
            zs_copy_select(L.k, false, fan_all, small, sh);
        }
        if (small) L.info.block = kSmallThreads;
#if defined(PURLIN_CHECKED)
        if ((h->inject == 2 || h->inject == 3) && p.nseg > 0) {
            // purlin_debug_inject: the first segment's destination (2) or
            // sources (3) one extent too far (every access past the call's
            // buffers is then skipped)
            if (h->inject == 2) {
                const int d = p.seg[0].dst == kEveryRank ? 0 : p.seg[0].dst;
                p.seg[0].dst_off += c.out_ext[d];
            } else {
                uint64_t ext = c.reduce ? 0 : c.in_ext[p.seg[0].src];
                for (int r = 0; c.reduce && r < c.R; ++r) ext = std::max(ext, c.in_ext[r]);
                p.seg[0].src_off += ext;
            }
            h->inject = 0;
        }
#endif
    }
    L.k.grid = (unsigned)grid;
    L.k.pdl = p.pdl != 0;
    L.kind = grid > 0 ? 1 : 0;
    L.info.chunk_bytes = tile_bytes(kn.max_unit_log2, kn.tile_units);
    L.info.grid = grid;
    L.info.kernels = grid > 0;
    return PURLIN_OK;
}

// Keep a recorded call as a plan (one call per plan).
purlin_status_t keep_plan(purlin_handle_t h, const Launches& L)
{
    if (h->recorded) return PURLIN_ERR_INVALID_ARG;
    purlin_plan* plan = new (std::nothrow) purlin_plan;
    if (!plan) return PURLIN_ERR_OOM;
    plan->h = h;
    plan->device = h->device;
    plan->kind = L.kind;
    auto keep = [](KernelLaunch& to, const KernelLaunch& from) {
        to.func = from.func;
        to.grid = from.grid;
        to.block = from.block;
        to.smem = from.smem;
        to.pdl = from.pdl;
        to.cooperative = from.cooperative;
        to.params_bytes = from.params_bytes;
        std::memcpy(to.params, from.params, from.params_bytes);
    };
    if (L.kind == 1 || L.kind == 3) keep(plan->k, L.k);
    if (L.kind == 3) keep(plan->k2, L.k2);
    plan->copies = L.copies;
    plan->info = L.info;
    h->recorded = plan;
    return PURLIN_OK;
}

// Launch what a call or a plan holds, in stream order.
cudaError_t launch_all(int kind, const KernelLaunch& k, const KernelLaunch& k2,
                       const std::vector<CopyOp>& copies, cudaStream_t s)
{
    cudaError_t ce = cudaSuccess;
    if (kind == 1 || kind == 3) {
        ce = launch_kernel(k, s);
        if (ce == cudaSuccess && kind == 3) ce = launch_kernel(k2, s);
    } else if (kind == 2) {
        for (const CopyOp& c : copies) {
            ce = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDefault, s);
            if (ce != cudaSuccess) break;
        }
    }
    return ce;
}

purlin_status_t run(purlin_handle_t h, Coll coll, const void* const in_[], void* const out_[],
                    const size_t* counts, const size_t* da, const size_t* db, size_t count,
                    int dtype, bool reduce, purlin_stream_t stream)
{
    if (!h || !in_ || !out_) return PURLIN_ERR_INVALID_ARG;
    if (coll != Coll::AllReduce && !counts) return PURLIN_ERR_INVALID_ARG;
    const size_t esz = elem_bytes(dtype);
    if (esz == 0) return PURLIN_ERR_INVALID_ARG;
    if (reduce && dtype == kU8) return PURLIN_ERR_UNSUPPORTED;
    const int R = h->R;

    uint64_t in[kMaxRanks], out[kMaxRanks];
    for (int r = 0; r < R; ++r) {
        in[r] = reinterpret_cast<uint64_t>(in_[r]);
        out[r] = reinterpret_cast<uint64_t>(out_[r]);
    }
    Piece pieces[kSegsLarge];
    int np = layout_pieces(coll, R, counts, da, db, count, esz, pieces, kSegsLarge);
    if (np < 0) return PURLIN_ERR_INVALID_ARG;
    uint64_t in_ext[kMaxRanks], out_ext[kMaxRanks];
    layout_extents(coll, R, counts, da, db, count, esz, in_ext, out_ext);
    purlin_status_t st = check_buffers(coll, R, in, out, in_ext, out_ext, esz, reduce, counts, da);
    if (st != PURLIN_OK) return st;
    if (coll == Coll::AllToAllV) {
        // received blocks inside one output must not overlap
        for (int a = 0; a < np; ++a)
            for (int b = a + 1; b < np; ++b)
                if (pieces[a].dst == pieces[b].dst &&
                    overlaps(pieces[a].dst_off, pieces[a].bytes, pieces[b].dst_off, pieces[b].bytes))
                    return PURLIN_ERR_INVALID_ARG;
    }

    DeviceGuard guard(h->device);
    if (!guard.ok) return PURLIN_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    purlin_launch_info_t info{};
    info.sms = h->sms;
    info.block = kThreads;
    info.bytes_moved = algorithmic_bytes(coll, R, counts, count, esz);

    // The call's launches are built in thread-local storage (no copy of a
    // parameter block on the way to the launch), then made at once or, while
    // a plan is being recorded, kept.
    static thread_local KernelLaunch tl_k, tl_k2;
    static thread_local std::vector<CopyOp> tl_copies;
    tl_k.grid = 0;
    tl_k2.grid = 0;
    tl_copies.clear();
    Launches L{tl_k, tl_k2, tl_copies, info};
    const CheckRanges check = call_ranges(R, in, out, in_ext, out_ext, violation_word(h->status));
    const Call c{h, coll, R, dtype, esz, reduce, in, out, pieces, np, &check, in_ext, out_ext};

    if (wants_staged(h) && np > 0) {
        st = plan_staged(c, L);
    } else {
        info.variant = PURLIN_VARIANT_ZS;
        // The TMA bulk Atom copies 16-byte aligned streams; a layout whose
        // sources and destinations sit on different alignments goes to the
        // vector kernels, whose shifted bodies realign it in registers.
        const bool bulk = !reduce && h->atom == PURLIN_ATOM_BULK &&
                          !needs_shift(pieces, np, R, in, out, esz, zs_knobs(h, coll, false));
        const ZsKnobs knobs = zs_knobs(h, coll, bulk);
        const bool by_destination =
            coll == Coll::AllToAllV ||
            (coll == Coll::AllGather &&
             (h->direction == PURLIN_DIRECTION_PULL ||
              (h->direction == PURLIN_DIRECTION_AUTO && !bulk && !outputs_share_grid(out, R))));
        if (!reduce && h->atom == PURLIN_ATOM_COPY_ENGINE)
            plan_copy_engine(c, L);
        else if (by_destination)
            st = plan_by_destination(c, knobs, bulk, L);
        else if (coll == Coll::AllReduce && np == 1 && R > 1 && !outputs_share_grid(out, R))
            st = plan_all_reduce_split(c, knobs, L);
        else
            st = plan_zs(c, knobs, bulk, L);
    }
    if (st != PURLIN_OK) return st;

    if (h->recording) return keep_plan(h, L);
    if (launch_all(L.kind, tl_k, tl_k2, tl_copies, s) != cudaSuccess) return PURLIN_ERR_CUDA;
    h->last = info;
    return PURLIN_OK;
}

}  // namespace

extern "C" {

int purlin_version(void) { return (kVersionMajor << 16) | kVersionMinor; }

const char* purlin_status_string(purlin_status_t s)
{
    switch (s) {
    case PURLIN_OK: return "ok";
    case PURLIN_ERR_INVALID_ARG: return "invalid argument";
    case PURLIN_ERR_UNSUPPORTED: return "unsupported request";
    case PURLIN_ERR_CUDA: return "CUDA runtime error";
    case PURLIN_ERR_TIMEOUT: return "device-side wait timed out";
    case PURLIN_ERR_OOM: return "device out of memory";
    case PURLIN_ERR_BOUNDS: return "an access outside the call's buffers was skipped";
    }
    return "unknown status";
}

purlin_status_t purlin_create(purlin_handle_t* out, int R, size_t staging_bytes, int device)
{
    if (!out) return PURLIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (R < 1 || R > PURLIN_MAX_RANKS || device < 0) return PURLIN_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return PURLIN_ERR_CUDA;
    if (device >= ndev) return PURLIN_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    if (!guard.ok) return PURLIN_ERR_CUDA;

    purlin_handle* h = new (std::nothrow) purlin_handle();
    if (!h) return PURLIN_ERR_OOM;
    h->R = R;
    h->device = device;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, device) != cudaSuccess) {
        delete h;
        return PURLIN_ERR_CUDA;
    }
    h->l2_bytes = (size_t)l2;
    h->staging_bytes = staging_bytes ? (staging_bytes + 255) & ~(size_t)255 : kDefaultStaging;
    h->flag_words = kFlagWords;
    if (cudaMalloc(&h->staging, h->staging_bytes) != cudaSuccess ||
        cudaMalloc(&h->flags, h->flag_words * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&h->status, kStatusBytes) != cudaSuccess) {
        cudaGetLastError();
        purlin_destroy(h);
        return PURLIN_ERR_OOM;
    }
    if (cudaMemset(h->flags, 0, h->flag_words * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(h->status, 0, kStatusBytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        purlin_destroy(h);
        return PURLIN_ERR_CUDA;
    }
    // Tuning knobs for measurements only; the defaults are the measured best.
    if (const char* u = std::getenv("PURLIN_PDL")) h->pdl = std::atoi(u) != 0;
    if (const char* u = std::getenv("PURLIN_L2_LOAD")) h->l2_load = std::atoi(u) % 3;
    {
        const char* names[4] = {"RS", "AG", "AR", "A2A"};
        char var[40];
        for (int i = 0; i < 4; ++i) {
            std::snprintf(var, sizeof var, "PURLIN_L2_%s_LOAD", names[i]);
            if (const char* u = std::getenv(var)) h->l2_coll_load[i] = std::atoi(u) % 3;
            std::snprintf(var, sizeof var, "PURLIN_L2_%s_STORE", names[i]);
            if (const char* u = std::getenv(var)) h->l2_coll_store[i] = std::atoi(u) % 3;
        }
    }
    if (const char* u = std::getenv("PURLIN_L2_STORE")) h->l2_store = std::atoi(u) % 3;
    if (const char* u = std::getenv("PURLIN_SMALL_TILES")) h->small_tiles = std::atol(u);
    if (const char* u = std::getenv("PURLIN_MAX_UNIT")) {
        const int v = std::atoi(u);
        for (int l = 1; l <= 5; ++l)
            if (v == (1 << l)) h->max_unit_log2 = l;
    }
    // The handle's initial policy, for sweeps: each value that purlin_set_policy
    // would accept replaces the default; anything else is ignored.
    if (const char* u = std::getenv("PURLIN_CHUNK")) {
        const long long v = std::atoll(u);
        if (v > 0 && v % 16 == 0) h->chunk_bytes = (size_t)v;
    }
    if (const char* u = std::getenv("PURLIN_DEPTH")) {
        const int v = std::atoi(u);
        if (v >= 1 && v <= 8) h->depth = v;
    }
    if (const char* u = std::getenv("PURLIN_CTAS")) {
        const int v = std::atoi(u);
        if (v >= 1 && v <= 65535) h->ctas = v;
    }
    if (const char* u = std::getenv("PURLIN_VARIANT")) {
        const int v = std::atoi(u);
        if (v >= PURLIN_VARIANT_AUTO && v <= PURLIN_VARIANT_STAGED_Y) h->variant = v;
    }
    *out = h;
    return PURLIN_OK;
}

purlin_status_t purlin_destroy(purlin_handle_t h)
{
    if (!h) return PURLIN_OK;
    delete h->recorded;  // a plan begun and never ended
    purlin_status_t st = PURLIN_OK;
    {
        DeviceGuard guard(h->device);
        if (cudaDeviceSynchronize() != cudaSuccess) st = PURLIN_ERR_CUDA;
        if (h->staging) cudaFree(h->staging);
        if (h->flags) cudaFree(h->flags);
        if (h->status) cudaFree(h->status);
    }
    delete h;
    return st;
}

purlin_status_t purlin_reduce_scatter(purlin_handle_t h, const void* const in[], void* const out[],
                                      const size_t recv_counts[], const size_t in_displs[],
                                      purlin_dtype_t dtype, purlin_op_t op, purlin_stream_t stream)
{
    if (op == PURLIN_OP_COPY) return PURLIN_ERR_UNSUPPORTED;
    if (op != PURLIN_OP_SUM) return PURLIN_ERR_INVALID_ARG;
    return run(h, Coll::ReduceScatter, in, out, recv_counts, in_displs, nullptr, 0, dtype, true,
               stream);
}

purlin_status_t purlin_all_gather(purlin_handle_t h, const void* const in[], void* const out[],
                                  const size_t counts[], const size_t out_displs[],
                                  purlin_dtype_t dtype, purlin_stream_t stream)
{
    return run(h, Coll::AllGather, in, out, counts, out_displs, nullptr, 0, dtype, false, stream);
}

purlin_status_t purlin_all_reduce(purlin_handle_t h, const void* const in[], void* const out[],
                                  size_t count, purlin_dtype_t dtype, purlin_op_t op,
                                  purlin_stream_t stream)
{
    if (op == PURLIN_OP_COPY) return PURLIN_ERR_UNSUPPORTED;
    if (op != PURLIN_OP_SUM) return PURLIN_ERR_INVALID_ARG;
    return run(h, Coll::AllReduce, in, out, nullptr, nullptr, nullptr, count, dtype, true, stream);
}

purlin_status_t purlin_all_to_all(purlin_handle_t h, const void* const in[], void* const out[],
                                  size_t count_per_pair, purlin_dtype_t dtype,
                                  purlin_stream_t stream)
{
    if (!h) return PURLIN_ERR_INVALID_ARG;
    size_t counts[kMaxRanks * kMaxRanks];
    for (int i = 0; i < h->R * h->R; ++i) counts[i] = count_per_pair;
    return run(h, Coll::AllToAllV, in, out, counts, nullptr, nullptr, 0, dtype, false, stream);
}

purlin_status_t purlin_all_to_all_v(purlin_handle_t h, const void* const in[], void* const out[],
                                    const size_t send_counts[], const size_t send_displs[],
                                    const size_t recv_displs[], purlin_dtype_t dtype,
                                    purlin_stream_t stream)
{
    return run(h, Coll::AllToAllV, in, out, send_counts, send_displs, recv_displs, 0, dtype, false,
               stream);
}

purlin_status_t purlin_set_policy(purlin_handle_t h, size_t chunk_bytes, int depth, int ctas,
                                  int variant)
{
    if (!h) return PURLIN_ERR_INVALID_ARG;
    if (chunk_bytes % 16 || depth < 0 || depth > 8 || ctas < 0 || ctas > 65535 ||
        variant < PURLIN_VARIANT_AUTO || variant > PURLIN_VARIANT_STAGED_Y)
        return PURLIN_ERR_INVALID_ARG;
    h->chunk_bytes = chunk_bytes;
    h->depth = depth;
    h->ctas = ctas;
    h->variant = variant;
    return PURLIN_OK;
}

purlin_status_t purlin_set_atom(purlin_handle_t h, int atom)
{
    if (!h || atom < PURLIN_ATOM_AUTO || atom > PURLIN_ATOM_COPY_ENGINE)
        return PURLIN_ERR_INVALID_ARG;
    h->atom = atom;
    return PURLIN_OK;
}

purlin_status_t purlin_set_direction(purlin_handle_t h, int direction)
{
    if (!h || direction < PURLIN_DIRECTION_AUTO || direction > PURLIN_DIRECTION_PULL)
        return PURLIN_ERR_INVALID_ARG;
    h->direction = direction;
    return PURLIN_OK;
}

purlin_status_t purlin_set_reduce_order(purlin_handle_t h, int order)
{
    if (!h || (order != PURLIN_ORDER_FIXED && order != PURLIN_ORDER_TREE))
        return PURLIN_ERR_INVALID_ARG;
    h->order = order;
    return PURLIN_OK;
}

purlin_status_t purlin_set_timeout(purlin_handle_t h, uint64_t timeout_ns)
{
    if (!h || timeout_ns == 0) return PURLIN_ERR_INVALID_ARG;
    h->timeout_ns = timeout_ns;
    return PURLIN_OK;
}

purlin_status_t purlin_plan_begin(purlin_handle_t h)
{
    if (!h || h->recording) return PURLIN_ERR_INVALID_ARG;
    h->recording = true;
    h->recorded = nullptr;
    return PURLIN_OK;
}

purlin_status_t purlin_plan_end(purlin_handle_t h, purlin_plan_t* plan)
{
    if (plan) *plan = nullptr;
    if (!h || !h->recording) return PURLIN_ERR_INVALID_ARG;
    h->recording = false;
    purlin_plan* rec = h->recorded;
    h->recorded = nullptr;
    if (!plan || !rec) {
        delete rec;
        return PURLIN_ERR_INVALID_ARG;
    }
    *plan = rec;
    return PURLIN_OK;
}

purlin_status_t purlin_plan_launch(purlin_plan_t plan, purlin_stream_t stream)
{
    if (!plan) return PURLIN_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return PURLIN_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_all(plan->kind, plan->k, plan->k2, plan->copies, s) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    plan->h->last = plan->info;
    return PURLIN_OK;
}

purlin_status_t purlin_plan_destroy(purlin_plan_t plan)
{
    delete plan;
    return PURLIN_OK;
}

purlin_status_t purlin_set_small_tiles(purlin_handle_t h, int tiles)
{
    if (!h || tiles < -1) return PURLIN_ERR_INVALID_ARG;
    h->small_tiles = tiles;
    return PURLIN_OK;
}

purlin_status_t purlin_debug_inject(purlin_handle_t h, int what)
{
    if (!h || what < 0 || what > 3) return PURLIN_ERR_INVALID_ARG;
#if !defined(PURLIN_CHECKED)
    if (what >= 2) return PURLIN_ERR_UNSUPPORTED;  // only a checked build catches it
#endif
    h->inject = what;
    return PURLIN_OK;
}

int purlin_debug_checked(void)
{
#if defined(PURLIN_CHECKED)
    return 1;
#else
    return 0;
#endif
}

purlin_status_t purlin_debug_violation(purlin_handle_t h, uint64_t* address)
{
    if (!h || !address) return PURLIN_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (!guard.ok) return PURLIN_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpy(&v, violation_word(h->status), sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (v != 0) {
        const unsigned long long zero = 0;
        if (cudaMemcpy(violation_word(h->status), &zero, sizeof zero, cudaMemcpyHostToDevice) !=
                cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return PURLIN_ERR_CUDA;
    }
    *address = (uint64_t)v;
    return PURLIN_OK;
}

purlin_status_t purlin_query_status(purlin_handle_t h)
{
    if (!h) return PURLIN_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    int v = 0;
    if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(h->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return PURLIN_ERR_CUDA;
    }
    return (purlin_status_t)v;
}

purlin_status_t purlin_last_launch(purlin_handle_t h, purlin_launch_info_t* info)
{
    if (!h || !info) return PURLIN_ERR_INVALID_ARG;
    *info = h->last;
    return PURLIN_OK;
}

purlin_status_t purlin_plan_segments(purlin_collective_t coll, int R, const uint64_t in_addr[],
                                     const uint64_t out_addr[], const size_t counts[],
                                     const size_t displs_a[], const size_t displs_b[],
                                     size_t count, purlin_dtype_t dtype, int max_unit,
                                     purlin_segment_t* segs, int max_segs, int* nsegs,
                                     uint32_t* ntiles)
{
    if (R < 1 || R > PURLIN_MAX_RANKS || !in_addr || !out_addr || !segs || !nsegs || !ntiles ||
        (max_unit != 16 && max_unit != 32) || coll < PURLIN_COLL_REDUCE_SCATTER ||
        coll > PURLIN_COLL_ALL_TO_ALL_V)
        return PURLIN_ERR_INVALID_ARG;
    Coll c = (Coll)coll;
    if (c != Coll::AllReduce && !counts) return PURLIN_ERR_INVALID_ARG;
    const size_t esz = elem_bytes(dtype);
    if (!esz) return PURLIN_ERR_INVALID_ARG;
    const bool reduce = c == Coll::ReduceScatter || c == Coll::AllReduce;
    if (reduce && dtype == PURLIN_U8) return PURLIN_ERR_UNSUPPORTED;
    for (int r = 0; r < R; ++r)
        if (reduce && (in_addr[r] % esz || out_addr[r] % esz)) return PURLIN_ERR_INVALID_ARG;
    Piece pieces[kSegsLarge];
    int np = layout_pieces(c, R, counts, displs_a, displs_b, count, esz, pieces, kSegsLarge);
    if (np < 0) return PURLIN_ERR_INVALID_ARG;
    Piece pulled[kMaxRanks * kMaxRanks];
    if (c == Coll::AllGather && !outputs_share_grid(out_addr, R)) {
        // as the launch (automatic direction): outputs on different 16-byte
        // alignments take the AllGather by destination
        np = pull_pieces(pieces, np, R, in_addr, out_addr, pulled);
        std::memcpy(pieces, pulled, sizeof(Piece) * (size_t)np);
    }
    Segment tmp[kSegsLarge];
    uint32_t nt = 0;
    const int tile_units = reduce ? kThreads * reduce_unroll(R, 0) : kTileUnitsCopy;
    int n = layout_segments(pieces, np, R, in_addr, out_addr, esz, reduce, tile_units,
                            max_unit == 32 ? 5 : 4, /*allow_shift=*/true, tmp, kSegsLarge, &nt);
    if (n > 0 && reduce && max_unit == 32) {
        bool shifted = false;   // as the launch: 16-byte bodies when a sum is shifted
        for (int i = 0; i < n; ++i) shifted |= tmp[i].shift != 0;
        if (shifted)
            n = layout_segments(pieces, np, R, in_addr, out_addr, esz, reduce, tile_units, 4,
                                /*allow_shift=*/true, tmp, kSegsLarge, &nt);
    }
    if (n < 0 || n > max_segs) return PURLIN_ERR_UNSUPPORTED;
    for (int i = 0; i < n; ++i) {
        segs[i].src_off = tmp[i].src_off;
        segs[i].dst_off = tmp[i].dst_off;
        segs[i].bytes = tmp[i].bytes;
        segs[i].src_rank = tmp[i].src == kEveryRank ? -1 : tmp[i].src;
        segs[i].dst_rank = tmp[i].dst == kEveryRank ? -1 : tmp[i].dst;
        segs[i].unit = 1 << tmp[i].unit_log2;
        segs[i].shift = tmp[i].shift & ~kShiftPerRank;
        segs[i].tile0 = tmp[i].tile0;
    }
    *nsegs = n;
    *ntiles = nt;
    return PURLIN_OK;
}

}  // extern "C"
