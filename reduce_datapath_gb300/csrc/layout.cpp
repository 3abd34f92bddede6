// layout.cpp -- the layout module: from a collective's naming of input and
// output partitions to the segments the Atom kernels execute.
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives":
//   - Abstract: collectives are "a naming of an input and output layout and a
//     copy or reduction operation"; coordination is derived from that naming.
//   - Figure 4: ReduceScatter sums partition k of every input into y_k at rank
//     k; AllGather places every y_k in rank order at every rank; AllToAll gives
//     rank j partition j of every source, in source order.
//   - Figure 6: AllReduce = AllGather composed with ReduceScatter.  Here its
//     zero-staging form fuses the two: each piece is summed once and written to
//     every output.
//   - Table 2: "(V)" variants take per-rank counts.
// Host code only; no CUDA calls.
#include "plan.h"

#include <algorithm>

namespace purlin {

namespace {

bool mul_ok(uint64_t a, uint64_t b, uint64_t* r)
{
    if (a != 0 && b > UINT64_MAX / a) return false;
    *r = a * b;
    return true;
}

bool add_ok(uint64_t a, uint64_t b, uint64_t* r)
{
    if (b > UINT64_MAX - a) return false;
    *r = a + b;
    return true;
}

// Start of partition k: displs[k], or the packed position.
uint64_t start_elem(const size_t* counts, const size_t* displs, int k, int stride = 1)
{
    if (displs) return displs[(size_t)k * stride];
    uint64_t s = 0;
    for (int m = 0; m < k; ++m) s += counts[(size_t)m * stride];
    return s;
}

int lowbit_log2(uint64_t v)
{
    int l = 0;
    while (l < 5 && !((v >> l) & 1u)) ++l;
    return l;
}

int log2_exact(uint64_t v)
{
    int l = 0;
    while (((uint64_t)1 << l) < v) ++l;
    return l;
}

}  // namespace

int layout_pieces(Coll coll, int R, const size_t* counts, const size_t* da, const size_t* db,
                  size_t count, size_t esz, Piece* out, int max_out)
{
    int n = 0;
    auto emit = [&](uint64_t src_e, uint64_t dst_e, uint64_t cnt, uint8_t src, uint8_t dst) {
        if (cnt == 0) return true;
        uint64_t so, dof, b;
        if (!mul_ok(src_e, esz, &so) || !mul_ok(dst_e, esz, &dof) || !mul_ok(cnt, esz, &b))
            return false;
        uint64_t end;
        if (!add_ok(so, b, &end) || !add_ok(dof, b, &end)) return false;
        if (n >= max_out) return false;
        out[n++] = Piece{so, dof, b, src, dst};
        return true;
    };
    switch (coll) {
    case Coll::ReduceScatter:
        // y_k = sum_r x_r[d_k : d_k + c_k]  ->  out[k][0 : c_k]
        for (int k = 0; k < R; ++k)
            if (!emit(start_elem(counts, da, k), 0, counts[k], kEveryRank, (uint8_t)k)) return -1;
        break;
    case Coll::AllGather:
        // in[k][0 : c_k]  ->  out[j][D_k : D_k + c_k] for every j
        for (int k = 0; k < R; ++k)
            if (!emit(0, start_elem(counts, da, k), counts[k], (uint8_t)k, kEveryRank)) return -1;
        break;
    case Coll::AllReduce:
        if (!emit(0, 0, count, kEveryRank, kEveryRank)) return -1;
        break;
    case Coll::AllToAllV:
        // in[s][sd[s][j] : + C[s][j]]  ->  out[j][rd[j][s] : + C[s][j]]
        for (int j = 0; j < R; ++j) {
            uint64_t packed_recv = 0;
            for (int s = 0; s < R; ++s) {
                uint64_t c = counts[(size_t)s * R + j];
                uint64_t sd = da ? da[(size_t)s * R + j] : start_elem(counts + (size_t)s * R, nullptr, j);
                uint64_t rd = db ? db[(size_t)j * R + s] : packed_recv;
                if (!emit(sd, rd, c, (uint8_t)s, (uint8_t)j)) return -1;
                packed_recv += c;
            }
        }
        break;
    }
    return n;
}

void layout_extents(Coll coll, int R, const size_t* counts, const size_t* da, const size_t* db,
                    size_t count, size_t esz, uint64_t in_ext[kMaxRanks], uint64_t out_ext[kMaxRanks])
{
    for (int r = 0; r < kMaxRanks; ++r) in_ext[r] = out_ext[r] = 0;
    switch (coll) {
    case Coll::ReduceScatter: {
        uint64_t hi = 0;
        for (int k = 0; k < R; ++k) {
            if (counts[k] == 0) continue;
            hi = std::max<uint64_t>(hi, (start_elem(counts, da, k) + counts[k]) * esz);
            out_ext[k] = (uint64_t)counts[k] * esz;
        }
        for (int r = 0; r < R; ++r) in_ext[r] = hi;
        break;
    }
    case Coll::AllGather: {
        uint64_t hi = 0;
        for (int k = 0; k < R; ++k) {
            in_ext[k] = (uint64_t)counts[k] * esz;
            if (counts[k]) hi = std::max<uint64_t>(hi, (start_elem(counts, da, k) + counts[k]) * esz);
        }
        for (int j = 0; j < R; ++j) out_ext[j] = hi;
        break;
    }
    case Coll::AllReduce:
        for (int r = 0; r < R; ++r) in_ext[r] = out_ext[r] = (uint64_t)count * esz;
        break;
    case Coll::AllToAllV:
        for (int j = 0; j < R; ++j) {
            uint64_t packed_recv = 0;
            for (int s = 0; s < R; ++s) {
                uint64_t c = counts[(size_t)s * R + j];
                uint64_t sd = da ? da[(size_t)s * R + j] : start_elem(counts + (size_t)s * R, nullptr, j);
                uint64_t rd = db ? db[(size_t)j * R + s] : packed_recv;
                packed_recv += c;
                if (!c) continue;
                in_ext[s] = std::max<uint64_t>(in_ext[s], (sd + c) * esz);
                out_ext[j] = std::max<uint64_t>(out_ext[j], (rd + c) * esz);
            }
        }
        break;
    }
}

int layout_segments(const Piece* pieces, int npieces, int R, const uint64_t* in_addr,
                    const uint64_t* out_addr, size_t esz, bool reduce, int tile_units,
                    int max_unit_log2, bool allow_shift, Segment* segs, int max_segs,
                    uint32_t* ntiles)
{
    int n = 0;
    uint64_t tiles = 0;
    const int elem_log2 = log2_exact(esz);
    auto push = [&](uint64_t so, uint64_t dof, uint64_t bytes, const Piece& p, int ulog2,
                    int shift = 0) {
        if (bytes == 0) return true;
        if (n >= max_segs) return false;
        Segment s{};
        s.src_off = so;
        s.dst_off = dof;
        s.bytes = bytes;
        s.src = p.src;
        s.dst = p.dst;
        s.unit_log2 = (uint8_t)ulog2;
        s.shift = (uint8_t)shift;
        s.tile0 = (uint32_t)tiles;
        uint64_t tb = tile_bytes(ulog2, shift ? shifted_tile_units(tile_units) : tile_units);
        tiles += (bytes + tb - 1) / tb;
        if (tiles > 0xffffffffull) return false;
        segs[n++] = s;
        return true;
    };
    auto same_residue = [](const uint64_t* a, int na, uint64_t mask) {
        for (int i = 1; i < na; ++i)
            if ((a[i] & mask) != (a[0] & mask)) return false;
        return true;
    };
    for (int i = 0; i < npieces; ++i) {
        const Piece& p = pieces[i];
        // Every address this piece touches, at its first byte: the sources
        // first (ns of them), then the destinations.
        uint64_t addrs[2 * kMaxRanks];
        int na = 0;
        if (p.src == kEveryRank)
            for (int r = 0; r < R; ++r) addrs[na++] = in_addr[r] + p.src_off;
        else
            addrs[na++] = in_addr[p.src] + p.src_off;
        const int ns = na;
        if (p.dst == kEveryRank)
            for (int r = 0; r < R; ++r) addrs[na++] = out_addr[r] + p.dst_off;
        else
            addrs[na++] = out_addr[p.dst] + p.dst_off;
        const uint64_t* dsts = addrs + ns;
        const int nd = na - ns;

        // Shifted body: the destinations agree on a vector alignment among
        // themselves but the sources do not share it.  The body's vector units
        // are aligned to the destinations (a head of less than one unit gets
        // there); every source is read from the unit boundary at or before it
        // and realigned in registers -- for a sum each rank on its own shift, so
        // its ranks' buffers may sit on different alignments.  Heads and tails
        // go element (sum) or byte-group (copy) wise.
        auto try_shifted = [&]() {
            // shifted sums take 16-byte units: with 32-byte ones the R blocks,
            // their neighbours' and the realignment outgrow the registers
            const int widest = reduce ? std::min(max_unit_log2, 4) : max_unit_log2;
            for (int u_log2 = widest; u_log2 >= 4; --u_log2) {
                const uint64_t u = (uint64_t)1 << u_log2, mask = u - 1;
                if (!same_residue(dsts, nd, mask)) continue;
                if (!reduce && !same_residue(addrs, ns, mask)) continue;
                const uint64_t head = std::min<uint64_t>((u - (dsts[0] & mask)) & mask, p.bytes);
                const uint64_t body = ((p.bytes - head) / u) * u;
                const uint64_t tail = p.bytes - head - body;
                // the first source off the destinations' grid (0: none is)
                int shift = 0;
                for (int a = 0; a < ns && shift == 0; ++a) shift = (int)((addrs[a] + head) & mask);
                if (body == 0 || shift == 0) return 0;
                if (!same_residue(addrs, ns, mask)) shift |= kShiftPerRank;
                // widest access every stream and the length allow, at offset `off`
                auto small_log2 = [&](uint64_t off, uint64_t len) {
                    if (reduce) return elem_log2;
                    uint64_t v = len;
                    for (int a = 0; a < na; ++a) v |= addrs[a] + off;
                    return std::min(lowbit_log2(v), max_unit_log2);
                };
                if (!push(p.src_off, p.dst_off, head, p, small_log2(0, head))) return -1;
                if (!push(p.src_off + head, p.dst_off + head, body, p, u_log2, shift)) return -1;
                if (!push(p.src_off + head + body, p.dst_off + head + body, tail, p,
                          small_log2(head + body, tail)))
                    return -1;
                return 1;
            }
            return 0;
        };

        // Widest unit at which all addresses share one residue: one common head
        // then aligns every stream at once.
        int body_log2 = -1;
        int min_body = reduce ? 4 : 0;  // sums vectorise at 16 or 32 bytes only
        for (int u = max_unit_log2; u >= min_body; --u) {
            uint64_t mask = ((uint64_t)1 << u) - 1;
            bool same = true;
            for (int a = 1; a < na; ++a) same &= ((addrs[a] & mask) == (addrs[0] & mask));
            if (same) { body_log2 = u; break; }
        }
        if (allow_shift && body_log2 < 4) {
            const int r = try_shifted();
            if (r < 0) return -1;
            if (r > 0) continue;
        }
        if (body_log2 < 0 || (reduce && body_log2 <= elem_log2)) {
            // Sums whose streams cannot share a vector alignment go element by element.
            if (!push(p.src_off, p.dst_off, p.bytes, p, reduce ? elem_log2 : 0)) return -1;
            continue;
        }
        uint64_t u = (uint64_t)1 << body_log2;
        uint64_t res = addrs[0] & (u - 1);
        uint64_t head = std::min<uint64_t>((u - res) & (u - 1), p.bytes);
        uint64_t body = ((p.bytes - head) / u) * u;
        uint64_t tail = p.bytes - head - body;
        int head_log2 = reduce ? elem_log2 : std::min(lowbit_log2(res), lowbit_log2(head));
        int tail_log2 = reduce ? elem_log2 : lowbit_log2(tail);
        if (!push(p.src_off, p.dst_off, head, p, head_log2)) return -1;
        if (!push(p.src_off + head, p.dst_off + head, body, p, body_log2)) return -1;
        if (!push(p.src_off + head + body, p.dst_off + head + body, tail, p, tail_log2)) return -1;
    }
    *ntiles = (uint32_t)tiles;
    return n;
}

}  // namespace purlin
