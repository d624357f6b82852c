// hc_sched.cpp -- host-side schedule generator of libhc.
//
// For each algorithm it lists, step by step, which rank's data flows where
// (the equivalent of the pages' per-rank link relations: CalcLinksRelation in
// the RHD article, CalcAGOmniPipeSliceInfo / OrchestrateLoop in the Pipeline
// article, the ring neighbour table of the Ring article), then binds every
// operand to the buffer that holds it at that step (input, working buffer or
// output) and cuts the work into loops.  The result is a list of kernel
// launches whose items the step kernel executes.
//
// Schedules (rank sets are rotations, see DevItem):
//  Ring ("Ring AllReduce带宽最优的环形流水线"; "AllReduce算法实现"):
//    reduce step s: rank q+1 computes  seg (q-s-1):  X_q-partial (+) own;
//    copy step s:   rank q+1 receives seg (q-s) from q.  Segment k's chain
//    starts at rank k+1 and ends at its owner k.
//  RHD (first article's RHD section; RHD article "算法描述", Table 1):
//    fold odd 2i+1 into even 2i (i < r = P - p'); over virtual ranks
//    (v = i for 2i, v = q - r for q >= 2r) exchange with v ^ d, d = 1, 2, ..
//    AllReduce halves a contiguous window (bit d clear keeps the low half)
//    and doubles it back; ReduceScatter / AllGather keep the blocks of the
//    virtual ranks that agree with v on the low bits (scatter order); the
//    folded ranks get their data last.
//  Pipeline ("HCCL Pipeline分级流水算法深度解析"): P = p_inter x p_intra,
//    rank = s * p_intra + l.  AllGather step t: (s,l) forwards the block of
//    (s-t+1, l) to (s+1, l) (t < p_inter) and to every (s, l'); the first
//    intra transfer rides in step 1, one lone intra step ends the phase.
//    ReduceScatter mirrors it: step 1 is a lone intra mesh reduce, step t
//    lets (s,l) mesh-reduce block (s-t, l) over its server (l, l+1, ...) and
//    fold in the partial arriving from (s-1, l).
#include <algorithm>
#include <cstring>
#include <map>
#include <set>
#include <tuple>

#include "hc_internal.h"

namespace hc {

namespace {

int pmod(int a, int m) { int r = a % m; return r < 0 ? r + m : r; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct RankSet {
    int base = 0, rot = 0, mod = 1, cnt = 0;
    int at(int i) const { return base + (rot + i) % mod; }
};
RankSet one(int r) { RankSet s; s.base = r; s.rot = 0; s.mod = 1; s.cnt = 1; return s; }
RankSet rotation(int base, int rot, int mod, int cnt) {
    RankSet s; s.base = base; s.rot = pmod(rot, mod); s.mod = mod; s.cnt = cnt; return s;
}

// Logical item: out[o] = (acc (+)) chain(ins) for each segment in segs.
struct LItem {
    RankSet outs;
    int acc = -1;
    RankSet ins;
    std::vector<int> segs;
};
using LStep = std::vector<LItem>;

std::vector<int> seg_range(int lo, int hi) {
    std::vector<int> v;
    for (int k = lo; k < hi; k++) v.push_back(k);
    return v;
}

int core_size(int P) { int q = 1; while (q * 2 <= P) q *= 2; return q; }

// ---------------------------------------------------------------- Ring
void ring_steps(hc_coll_t coll, int P, std::vector<LStep>& st) {
    if (coll != HC_COLL_ALLGATHER) {
        for (int s = 0; s + 1 < P; s++) {
            LStep x;
            for (int q = 0; q < P; q++) {
                int d = (q + 1) % P;
                LItem it;
                it.outs = one(d);
                it.acc = q;
                it.ins = one(d);
                it.segs = {pmod(q - s - 1, P)};
                x.push_back(it);
            }
            st.push_back(x);
        }
    }
    if (coll != HC_COLL_REDUCE_SCATTER) {
        for (int s = 0; s + 1 < P; s++) {
            LStep x;
            for (int q = 0; q < P; q++) {
                LItem it;
                it.outs = one((q + 1) % P);
                it.ins = one(q);
                it.segs = {pmod(q - s, P)};
                x.push_back(it);
            }
            st.push_back(x);
        }
    }
}

// ---------------------------------------------------------------- RHD
void rhd_steps(hc_coll_t coll, int P, std::vector<LStep>& st) {
    const int pp = core_size(P);
    const int r = P - pp;
    auto real = [r](int v) { return v < r ? 2 * v : v + r; };
    // real blocks owned by virtual rank w (scatter order)
    auto blocks_of = [r](int w, std::vector<int>& out) {
        if (w < r) { out.push_back(2 * w); out.push_back(2 * w + 1); }
        else out.push_back(w + r);
    };
    auto fold_step = [&](int nseg) {
        LStep x;
        for (int i = 0; i < r; i++) {
            LItem it;
            it.outs = one(2 * i);
            it.acc = 2 * i + 1;
            it.ins = one(2 * i);
            it.segs = seg_range(0, nseg);
            x.push_back(it);
        }
        st.push_back(x);
    };

    if (coll == HC_COLL_ALLREDUCE) {
        const int S = pp;
        if (r) fold_step(S);
        std::vector<int> wlo(pp, 0), whi(pp, S);
        for (int d = 1; d < pp; d <<= 1) {
            LStep x;
            std::vector<int> nlo(pp), nhi(pp);
            for (int v = 0; v < pp; v++) {
                int u = v ^ d, mid = (wlo[v] + whi[v]) / 2;
                bool low = (v & d) == 0;
                int glo = low ? mid : wlo[v], ghi = low ? whi[v] : mid;  // half v gives away
                nlo[v] = low ? wlo[v] : mid;
                nhi[v] = low ? mid : whi[v];
                LItem it;
                it.outs = one(real(u));
                it.acc = real(v);
                it.ins = one(real(u));
                it.segs = seg_range(glo, ghi);
                x.push_back(it);
            }
            wlo = nlo; whi = nhi;
            st.push_back(x);
        }
        for (int d = pp / 2; d >= 1; d >>= 1) {
            LStep x;
            std::vector<int> nlo(pp), nhi(pp);
            for (int v = 0; v < pp; v++) {
                int u = v ^ d;
                LItem it;
                it.outs = one(real(u));
                it.ins = one(real(v));
                it.segs = seg_range(wlo[v], whi[v]);
                x.push_back(it);
                nlo[v] = std::min(wlo[v], wlo[u]);
                nhi[v] = std::max(whi[v], whi[u]);
            }
            wlo = nlo; whi = nhi;
            st.push_back(x);
        }
        if (r) {
            LStep x;
            for (int i = 0; i < r; i++) {
                LItem it;
                it.outs = one(2 * i + 1);
                it.ins = one(2 * i);
                it.segs = seg_range(0, S);
                x.push_back(it);
            }
            st.push_back(x);
        }
        return;
    }
    if (coll == HC_COLL_REDUCE_SCATTER) {
        if (r) fold_step(P);
        for (int d = 1; d < pp; d <<= 1) {
            LStep x;
            for (int v = 0; v < pp; v++) {
                int u = v ^ d;
                LItem it;
                it.outs = one(real(u));
                it.acc = real(v);
                it.ins = one(real(u));
                for (int w = 0; w < pp; w++)
                    if ((w & (d - 1)) == (v & (d - 1)) && (w & d) == (u & d)) blocks_of(w, it.segs);
                std::sort(it.segs.begin(), it.segs.end());
                x.push_back(it);
            }
            st.push_back(x);
        }
        if (r) {
            LStep x;
            for (int i = 0; i < r; i++) {
                LItem it;
                it.outs = one(2 * i + 1);
                it.ins = one(2 * i);
                it.segs = {2 * i + 1};
                x.push_back(it);
            }
            st.push_back(x);
        }
        return;
    }
    // AllGather: mirror of the ReduceScatter
    if (r) {
        LStep x;
        for (int i = 0; i < r; i++) {
            LItem it;
            it.outs = one(2 * i);
            it.ins = one(2 * i + 1);
            it.segs = {2 * i + 1};
            x.push_back(it);
        }
        st.push_back(x);
    }
    for (int d = pp / 2; d >= 1; d >>= 1) {
        LStep x;
        for (int v = 0; v < pp; v++) {
            int u = v ^ d;
            LItem it;
            it.outs = one(real(u));
            it.ins = one(real(v));
            for (int w = 0; w < pp; w++)
                if ((w & (2 * d - 1)) == (v & (2 * d - 1))) blocks_of(w, it.segs);
            std::sort(it.segs.begin(), it.segs.end());
            x.push_back(it);
        }
        st.push_back(x);
    }
    if (r) {
        LStep x;
        for (int i = 0; i < r; i++) {
            LItem it;
            it.outs = one(2 * i + 1);
            it.ins = one(2 * i);
            it.segs = seg_range(0, P);
            x.push_back(it);
        }
        st.push_back(x);
    }
}

// ---------------------------------------------------------------- Pipeline
void pipe_steps(hc_coll_t coll, int P, int pin, std::vector<LStep>& st) {
    const int pout = P / pin;
    auto rank = [pin](int s, int l) { return s * pin + l; };
    if (coll != HC_COLL_ALLGATHER) {
        for (int t = 1; t <= pout; t++) {
            if (t == 1 && pin == 1) continue;  // a lone intra step with one rank per server is empty
            LStep x;
            for (int s = 0; s < pout; s++)
                for (int l = 0; l < pin; l++) {
                    LItem it;
                    it.outs = one(rank(s, l));
                    it.acc = t >= 2 ? rank(pmod(s - 1, pout), l) : -1;
                    it.ins = rotation(s * pin, l, pin, pin);
                    it.segs = {rank(pmod(s - t, pout), l)};
                    x.push_back(it);
                }
            st.push_back(x);
        }
    }
    if (coll != HC_COLL_REDUCE_SCATTER) {
        for (int t = 1; t <= pout; t++) {
            LStep x;
            for (int s = 0; s < pout; s++)
                for (int l = 0; l < pin; l++) {
                    int blk = rank(pmod(s - t + 1, pout), l);
                    if (t <= pout - 1) {
                        LItem it;
                        it.outs = one(rank((s + 1) % pout, l));
                        it.ins = one(rank(s, l));
                        it.segs = {blk};
                        x.push_back(it);
                    }
                    if (pin > 1) {
                        LItem it;
                        it.outs = rotation(s * pin, l + 1, pin, pin - 1);
                        it.ins = one(rank(s, l));
                        it.segs = {blk};
                        x.push_back(it);
                    }
                }
            if (!x.empty()) st.push_back(x);
        }
    }
}

// ---------------------------------------------------------------- Broadcast
// RHD Broadcast: part1 members of the root's parity join the power-of-two
// block, distance halving spreads the vector (partner v ^ p'/2, ..., v ^ 1),
// then each part1 member sends it to its pair partner.
void rhd_bcast_steps(int P, int root, std::vector<LStep>& st) {
    const int pp = core_size(P);
    const int r = P - pp;
    const int par = root & 1;
    auto real = [r, par](int v) { return v < r ? 2 * v + par : v + r; };
    std::vector<char> have(pp, 0);
    have[root < 2 * r ? root / 2 : root - r] = 1;
    for (int d = pp / 2; d >= 1; d >>= 1) {
        LStep x;
        std::vector<char> nxt = have;
        for (int v = 0; v < pp; v++) {
            if (!have[v]) continue;
            LItem it;
            it.outs = one(real(v ^ d));
            it.ins = one(real(v));
            it.segs = {0};
            x.push_back(it);
            nxt[v ^ d] = 1;
        }
        have = nxt;
        st.push_back(x);
    }
    if (r) {
        LStep x;
        for (int i = 0; i < r; i++) {
            LItem it;
            it.outs = one(2 * i + 1 - par);
            it.ins = one(2 * i + par);
            it.segs = {0};
            x.push_back(it);
        }
        st.push_back(x);
    }
}

// ---------------------------------------------------------------- hierarchical
// Plain hierarchical AllReduce: mesh ReduceScatter inside each server, RHD
// AllReduce among equal local indices across servers on intra segment l
// (segments l*p' .. l*p' + p' - 1), mesh AllGather inside each server.
void hier_steps(int P, int pin, std::vector<LStep>& st) {
    const int pout = P / pin;
    const int pp = core_size(pout);
    const int r = pout - pp;
    auto sv = [r](int v) { return v < r ? 2 * v : v + r; };  // virtual -> real server
    auto intra_seg = [pp](int l) { return seg_range(l * pp, (l + 1) * pp); };
    if (pin > 1) {
        LStep x;
        for (int s = 0; s < pout; s++)
            for (int l = 0; l < pin; l++) {
                LItem it;
                it.outs = one(s * pin + l);
                it.ins = rotation(s * pin, l, pin, pin);
                it.segs = intra_seg(l);
                x.push_back(it);
            }
        st.push_back(x);
    }
    if (r) {
        LStep x;
        for (int l = 0; l < pin; l++)
            for (int i = 0; i < r; i++) {
                LItem it;
                it.outs = one(2 * i * pin + l);
                it.acc = (2 * i + 1) * pin + l;
                it.ins = one(2 * i * pin + l);
                it.segs = intra_seg(l);
                x.push_back(it);
            }
        st.push_back(x);
    }
    std::vector<int> wlo(pp, 0), whi(pp, pp);
    for (int d = 1; d < pp; d <<= 1) {
        LStep x;
        std::vector<int> nlo(pp), nhi(pp);
        for (int v = 0; v < pp; v++) {
            const int u = v ^ d, mid = (wlo[v] + whi[v]) / 2;
            const bool low = (v & d) == 0;
            const int glo = low ? mid : wlo[v], ghi = low ? whi[v] : mid;
            nlo[v] = low ? wlo[v] : mid;
            nhi[v] = low ? mid : whi[v];
            for (int l = 0; l < pin; l++) {
                LItem it;
                it.outs = one(sv(u) * pin + l);
                it.acc = sv(v) * pin + l;
                it.ins = one(sv(u) * pin + l);
                it.segs = seg_range(l * pp + glo, l * pp + ghi);
                x.push_back(it);
            }
        }
        wlo = nlo;
        whi = nhi;
        st.push_back(x);
    }
    for (int d = pp / 2; d >= 1; d >>= 1) {
        LStep x;
        std::vector<int> nlo(pp), nhi(pp);
        for (int v = 0; v < pp; v++) {
            const int u = v ^ d;
            for (int l = 0; l < pin; l++) {
                LItem it;
                it.outs = one(sv(u) * pin + l);
                it.ins = one(sv(v) * pin + l);
                it.segs = seg_range(l * pp + wlo[v], l * pp + whi[v]);
                x.push_back(it);
            }
            nlo[v] = std::min(wlo[v], wlo[u]);
            nhi[v] = std::max(whi[v], whi[u]);
        }
        wlo = nlo;
        whi = nhi;
        st.push_back(x);
    }
    if (r) {
        LStep x;
        for (int l = 0; l < pin; l++)
            for (int i = 0; i < r; i++) {
                LItem it;
                it.outs = one((2 * i + 1) * pin + l);
                it.ins = one(2 * i * pin + l);
                it.segs = intra_seg(l);
                x.push_back(it);
            }
        st.push_back(x);
    }
    if (pin > 1) {
        LStep x;
        for (int s = 0; s < pout; s++)
            for (int l = 0; l < pin; l++) {
                LItem it;
                it.outs = rotation(s * pin, l + 1, pin, pin - 1);
                it.ins = one(s * pin + l);
                it.segs = intra_seg(l);
                x.push_back(it);
            }
        st.push_back(x);
    }
}

bool logical_steps(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root,
                   std::vector<LStep>& st) {
    st.clear();
    if (algo == HC_ALGO_HIER) {
        if (coll != HC_COLL_ALLREDUCE || p_intra < 1 || P % p_intra) return false;
        hier_steps(P, p_intra, st);
        return true;
    }
    if (coll == HC_COLL_BROADCAST) {
        if (algo != HC_ALGO_RHD || root < 0 || root >= P) return false;
        rhd_bcast_steps(P, root, st);
        return true;
    }
    if (algo == HC_ALGO_RING) ring_steps(coll, P, st);
    else if (algo == HC_ALGO_RHD) rhd_steps(coll, P, st);
    else if (algo == HC_ALGO_PIPELINE) {
        if (p_intra < 1 || P % p_intra) return false;
        pipe_steps(coll, P, p_intra, st);
    } else return false;
    return true;
}

// Split a sorted segment list into strided runs (first, width, stride, reps).
struct SegPattern { int first, width, stride, reps; };
std::vector<SegPattern> encode_segments(const std::vector<int>& segs) {
    std::vector<std::pair<int, int>> runs;  // (start, length)
    for (size_t i = 0; i < segs.size();) {
        size_t j = i + 1;
        while (j < segs.size() && segs[j] == segs[j - 1] + 1) j++;
        runs.push_back({segs[i], (int)(j - i)});
        i = j;
    }
    std::vector<SegPattern> out;
    for (size_t i = 0; i < runs.size();) {
        SegPattern p{runs[i].first, runs[i].second, runs[i].second, 1};
        size_t j = i + 1;
        if (j < runs.size() && runs[j].second == p.width) {
            p.stride = runs[j].first - runs[i].first;
            p.reps = 2;
            j++;
            while (j < runs.size() && runs[j].second == p.width &&
                   runs[j].first - runs[j - 1].first == p.stride) {
                p.reps++;
                j++;
            }
        }
        out.push_back(p);
        i = j;
    }
    return out;
}

constexpr uint8_t LOC_NONE = 255;

DevItem make_item(const RankSet& outs, uint8_t out_loc, int acc, uint8_t acc_loc,
                  const RankSet& ins, uint8_t in_loc, const SegPattern& sp) {
    DevItem d;
    std::memset(&d, 0, sizeof d);
    d.out_base = (int16_t)outs.base; d.out_rot = (int16_t)outs.rot;
    d.out_mod = (int16_t)outs.mod;   d.out_cnt = (int16_t)outs.cnt;
    d.in_base = (int16_t)ins.base;   d.in_rot = (int16_t)ins.rot;
    d.in_mod = (int16_t)ins.mod;     d.in_cnt = (int16_t)ins.cnt;
    d.acc_rank = (int16_t)acc;
    d.acc_loc = acc >= 0 ? acc_loc : 0;
    d.in_loc = in_loc;
    d.out_loc = out_loc;
    d.seg_width = (int16_t)sp.width;
    d.seg_reps = (int16_t)sp.reps;
    d.seg_first = sp.first;
    d.seg_stride = sp.stride;
    d.out2_mod = 1;  // empty second output set
    return d;
}

// Merge copies of one step that read the same input block (same location,
// rank and segments) and write the same location: the second's outputs
// become the first's second output set, so the block is read once.
void merge_copies(std::vector<DevItem>& items) {
    std::vector<DevItem> out;
    std::vector<char> taken(items.size(), 0);
    for (size_t i = 0; i < items.size(); i++) {
        if (taken[i]) continue;
        DevItem a = items[i];
        const bool copy = a.in_cnt == 1 && a.acc_rank < 0;
        for (size_t j = i + 1; copy && a.out2_cnt == 0 && j < items.size(); j++) {
            const DevItem& b = items[j];
            if (taken[j] || b.in_cnt != 1 || b.acc_rank >= 0 || b.out2_cnt != 0) continue;
            if (b.in_loc != a.in_loc || b.out_loc != a.out_loc) continue;
            if (b.in_base + b.in_rot % b.in_mod != a.in_base + a.in_rot % a.in_mod) continue;
            if (b.seg_first != a.seg_first || b.seg_width != a.seg_width ||
                b.seg_reps != a.seg_reps || (a.seg_reps > 1 && b.seg_stride != a.seg_stride))
                continue;
            a.out2_base = b.out_base;
            a.out2_rot = b.out_rot;
            a.out2_mod = b.out_mod;
            a.out2_cnt = b.out_cnt;
            taken[j] = 1;
        }
        out.push_back(a);
    }
    items.swap(out);
}

}  // namespace

// ---------------------------------------------------------------------------
int num_segments(hc_algo_t algo, hc_coll_t coll, int P, int p_intra) {
    if (P < 1) return 0;
    if (coll == HC_COLL_BROADCAST) return 1;
    if (algo == HC_ALGO_HIER) {
        if (p_intra < 1 || P % p_intra) return 0;
        return p_intra * core_size(P / p_intra);
    }
    if (algo == HC_ALGO_RHD && coll == HC_COLL_ALLREDUCE) return core_size(P);
    return P;
}

Layout make_layout(hc_algo_t algo, hc_coll_t coll, int P, int64_t n, hc_dtype_t dt, int p_intra) {
    Layout lay;
    lay.S = num_segments(algo, coll, P, p_intra);
    lay.n = n;
    lay.A = kVecBytes / elem_bytes(dt);
    lay.L = (lay.S > 0 && n > 0) ? cdiv(cdiv(n, lay.S), lay.A) * lay.A : 0;
    return lay;
}

// Loop slicer: c = align_down(loop_bytes / (P * slots * b), 128 / b).
Slicing make_slicing(hc_algo_t algo, int P, int p_intra, const Layout& lay, hc_dtype_t dt,
                     int64_t loop_bytes) {
    Slicing s;
    s.chunk = lay.L;
    s.loops = 1;
    s.tail = lay.L;
    if (lay.L <= 0 || loop_bytes <= 0) return s;
    const int64_t b = elem_bytes(dt);
    int64_t slots = 1;
    if (algo == HC_ALGO_RHD) slots = (P + 1) / 2;
    else if (algo == HC_ALGO_PIPELINE || algo == HC_ALGO_HIER) slots = std::max(1, p_intra - 1);
    const int64_t granule = 128 / b;
    int64_t c = loop_bytes / ((int64_t)P * slots * b);
    c -= c % granule;
    if (c < granule) c = granule;
    if (c >= lay.L) return s;
    s.chunk = c;
    s.loops = (int)cdiv(lay.L, c);
    s.tail = lay.L - (int64_t)(s.loops - 1) * c;
    return s;
}

bool build_plan(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root, int64_t n,
                hc_dtype_t dt, int64_t loop_bytes, const Aliasing& alias, Plan* out) {
    if (P < 1 || P > kMaxRanks || n < 0) return false;
    std::vector<LStep> steps;
    if (!logical_steps(algo, coll, P, p_intra, root, steps)) return false;
    Plan& plan = *out;
    plan = Plan();
    plan.lay = make_layout(algo, coll, P, n, dt, p_intra);
    plan.sl = make_slicing(algo, P, p_intra, plan.lay, dt, loop_bytes);
    plan.steps_per_loop = (int)steps.size();
    const int S = plan.lay.S;

    // where each (rank, segment) currently lives
    std::vector<uint8_t> state((size_t)P * S, LOC_ORIG);
    if (coll == HC_COLL_ALLGATHER) {
        std::fill(state.begin(), state.end(), LOC_NONE);
        for (int q = 0; q < P; q++) state[(size_t)q * S + q] = LOC_ORIG;
    }
    if (coll == HC_COLL_BROADCAST) {
        std::fill(state.begin(), state.end(), LOC_NONE);
        state[(size_t)root * S] = LOC_ORIG;
    }
    auto st_at = [&](int q, int k) -> uint8_t& { return state[(size_t)q * S + k]; };

    // bind one loop's steps to buffer locations
    std::vector<std::vector<DevItem>> bound;
    for (size_t si = 0; si < steps.size(); si++) {
        std::vector<DevItem> items;
        if (si == 0 && coll == HC_COLL_ALLGATHER) {
            // LocalCopy of the own block, only where input and output differ;
            // it reads the input, which nothing in this step writes
            for (int q = 0; q < P; q++)
                if (!alias.orig_is_work[q])
                    items.push_back(make_item(one(q), LOC_WORK, -1, 0, one(q), LOC_ORIG,
                                              SegPattern{q, 1, 1, 1}));
        }
        if (si == 0 && coll == HC_COLL_BROADCAST && !alias.orig_is_work[root])
            items.push_back(make_item(one(root), LOC_WORK, -1, 0, one(root), LOC_ORIG,
                                      SegPattern{0, 1, 1, 1}));
        for (const LItem& li : steps[si]) {
            // group segments by the locations of their operands
            std::map<std::pair<int, int>, std::vector<int>> groups;
            for (int k : li.segs) {
                uint8_t al = li.acc >= 0 ? st_at(li.acc, k) : 0;
                uint8_t il = st_at(li.ins.at(0), k);
                for (int i = 1; i < li.ins.cnt; i++)
                    if (st_at(li.ins.at(i), k) != il) return false;  // not produced by these schedules
                if (il == LOC_NONE || al == LOC_NONE) return false;
                groups[{al, il}].push_back(k);
            }
            for (auto& g : groups)
                for (const SegPattern& sp : encode_segments(g.second))
                    items.push_back(make_item(li.outs, LOC_WORK, li.acc, (uint8_t)g.first.first,
                                              li.ins, (uint8_t)g.first.second, sp));
        }
        for (const LItem& li : steps[si])
            for (int o = 0; o < li.outs.cnt; o++)
                for (int k : li.segs) st_at(li.outs.at(o), k) = LOC_WORK;
        if (si == 0 && coll == HC_COLL_ALLGATHER)
            for (int q = 0; q < P; q++) st_at(q, q) = LOC_WORK;
        if (si == 0 && coll == HC_COLL_BROADCAST) st_at(root, 0) = LOC_WORK;
        merge_copies(items);
        bound.push_back(items);
    }

    // results that must still be moved into place (full segments, one launch)
    std::vector<DevItem> final_items;
    if (coll == HC_COLL_REDUCE_SCATTER) {
        for (int q = 0; q < P; q++)
            if (!alias.final_is_work[q])
                final_items.push_back(make_item(one(q), LOC_FINAL, -1, 0, one(q), st_at(q, q),
                                                SegPattern{q, 1, 1, 1}));
    } else {
        for (int q = 0; q < P; q++) {
            std::vector<int> pending;
            for (int k = 0; k < S; k++) {
                if (st_at(q, k) == LOC_NONE) return false;  // a block never delivered
                if (st_at(q, k) == LOC_ORIG && !alias.orig_is_work[q]) pending.push_back(k);
            }
            for (const SegPattern& sp : encode_segments(pending))
                final_items.push_back(make_item(one(q), LOC_WORK, -1, 0, one(q), LOC_ORIG, sp));
        }
    }

    // inputs no launch of this call writes: the original buffers of ranks
    // that are out of place (every output goes to LOC_WORK or LOC_FINAL)
    auto mark_early = [&](std::vector<DevItem>& items) {
        for (DevItem& it : items) {
            bool ok = it.in_loc == LOC_ORIG;
            for (int j = 0; ok && j < it.in_cnt; j++)
                ok = !alias.orig_is_work[it.in_base + (it.in_rot + j) % it.in_mod];
            it.early = ok ? 1 : 0;
        }
    };
    for (auto& items : bound) mark_early(items);
    mark_early(final_items);

    // operands read by one item of a launch only: the kernels load them with
    // an L2 evict-first policy (what stays in L2 is then what later steps
    // read again); an operand two items read (the Pipeline AllGather forwards
    // a block and broadcasts it in the same step) keeps the normal policy
    auto mark_once = [&](std::vector<DevItem>& items) {
        std::map<std::tuple<int, int, int>, int> reads;  // (location, rank, segment) -> items
        auto each = [&](const DevItem& it, auto&& fn) {
            for (int i = 0; i < it.seg_width * it.seg_reps; i++) {
                const int k = it.seg_first + (i / it.seg_width) * it.seg_stride + i % it.seg_width;
                for (int j = 0; j < it.in_cnt; j++)
                    fn(std::make_tuple((int)it.in_loc, it.in_base + (it.in_rot + j) % it.in_mod, k));
                if (it.acc_rank >= 0) fn(std::make_tuple((int)it.acc_loc, (int)it.acc_rank, k));
            }
        };
        for (const DevItem& it : items) each(it, [&](const std::tuple<int, int, int>& t) { reads[t]++; });
        for (DevItem& it : items) {
            bool once = true;
            each(it, [&](const std::tuple<int, int, int>& t) { once = once && reads[t] == 1; });
            it.once = once ? 1 : 0;
        }
    };
    for (auto& items : bound) mark_once(items);
    mark_once(final_items);

    // outputs a later launch of the call reads: within a loop, a later step
    // or the final moves (each loop acts on its own slice, so only the steps
    // after this one in the same loop see its output); an in-place rank's
    // original buffer is its working buffer, and so is an in-place
    // ReduceScatter's output segment
    auto canon = [&](int loc, int q, int k) {
        if ((loc == LOC_ORIG && alias.orig_is_work[q]) || (loc == LOC_FINAL && alias.final_is_work[q]))
            loc = LOC_WORK;
        return std::make_tuple(loc, q, k);
    };
    std::set<std::tuple<int, int, int>> read_later;
    auto note_reads = [&](const std::vector<DevItem>& items) {
        for (const DevItem& it : items)
            for (int i = 0; i < it.seg_width * it.seg_reps; i++) {
                const int k = it.seg_first + (i / it.seg_width) * it.seg_stride + i % it.seg_width;
                for (int j = 0; j < it.in_cnt; j++)
                    read_later.insert(canon(it.in_loc, it.in_base + (it.in_rot + j) % it.in_mod, k));
                if (it.acc_rank >= 0) read_later.insert(canon(it.acc_loc, it.acc_rank, k));
            }
    };
    auto set_read_later = [&](const DevItem& it, int base, int rot, int mod, int cnt) {
        for (int i = 0; i < it.seg_width * it.seg_reps; i++) {
            const int k = it.seg_first + (i / it.seg_width) * it.seg_stride + i % it.seg_width;
            for (int j = 0; j < cnt; j++)
                if (read_later.count(canon(it.out_loc, base + (rot + j) % mod, k))) return true;
        }
        return false;
    };
    note_reads(final_items);  // the final moves' outputs are read by nobody
    for (size_t si = bound.size(); si-- > 0;) {
        for (DevItem& it : bound[si])
            it.keep = (uint8_t)((set_read_later(it, it.out_base, it.out_rot, it.out_mod, it.out_cnt) ? 1 : 0) |
                                (set_read_later(it, it.out2_base, it.out2_rot, it.out2_mod, it.out2_cnt) ? 2 : 0));
        note_reads(bound[si]);
    }

    if (plan.lay.n == 0) return true;
    for (int lp = 0; lp < plan.sl.loops; lp++) {
        int64_t lo = (int64_t)lp * plan.sl.chunk;
        int64_t hi = std::min(lo + plan.sl.chunk, plan.lay.L);
        for (size_t si = 0; si < bound.size(); si++) {
            if (bound[si].empty()) continue;
            PlanLaunch L;
            L.lo = lo;
            L.hi = hi;
            L.items = bound[si];
            L.step = (int)si;
            L.loop = lp;
            plan.launches.push_back(L);
        }
    }
    if (!final_items.empty()) {
        PlanLaunch L;
        L.lo = 0;
        L.hi = plan.lay.L;
        L.items = final_items;
        L.step = (int)bound.size();
        L.loop = -1;
        plan.launches.push_back(L);
    }
    return true;
}

bool schedule_traffic(hc_algo_t algo, hc_coll_t coll, int P, int p_intra, int root, int64_t n,
                      hc_dtype_t dt, int64_t loop_bytes, int* steps_per_loop,
                      unsigned long long* bytes_sent) {
    std::vector<LStep> steps;
    if (P < 1 || P > kMaxRanks || !logical_steps(algo, coll, P, p_intra, root, steps)) return false;
    (void)loop_bytes;
    Layout lay = make_layout(algo, coll, P, n, dt, p_intra);
    const int b = elem_bytes(dt);
    if (steps_per_loop) *steps_per_loop = (int)steps.size();
    if (!bytes_sent) return true;
    for (int q = 0; q < P; q++) bytes_sent[q] = 0;
    for (const LStep& x : steps)
        for (const LItem& li : x)
            for (int k : li.segs) {
                unsigned long long len = (unsigned long long)(lay.seg_hi(k) - lay.seg_lo(k)) * b;
                for (int o = 0; o < li.outs.cnt; o++) {
                    int dst = li.outs.at(o);
                    if (li.acc >= 0 && li.acc != dst) bytes_sent[li.acc] += len;
                    for (int i = 0; i < li.ins.cnt; i++)
                        if (li.ins.at(i) != dst) bytes_sent[li.ins.at(i)] += len;
                }
            }
    return true;
}

// Vectors an item processes in a launch (upper bound: full-length segments).
static int64_t item_vectors(const DevItem& it, const PlanLaunch& L, const Layout& lay) {
    int64_t v = cdiv(L.hi - L.lo, lay.A);
    return v * (int64_t)it.seg_width * it.seg_reps;
}

// CTAs per item: one per `threads` vectors when the budget allows; otherwise
// the budget is shared in proportion to the bytes each item moves (vectors x
// its inputs, accumulator and outputs), so that items of one launch finish
// together; and never fewer than the item's segments.  (Shared by vectors alone, a Pipeline AllGather step whose 1 -> 7
// broadcast items sit beside 1 -> 1 forwards gave both kinds the same CTAs
// and ran at 0.68 of the copy bandwidth on GB300.)
int assign_ctas(PlanLaunch& L, const Layout& lay, int threads, int max_ctas) {
    const int ni = (int)L.items.size();
    if (ni == 0) return 0;
    std::vector<int64_t> need(ni), weight(ni);
    int64_t total = 0, wsum = 0;
    for (int i = 0; i < ni; i++) {
        const DevItem& it = L.items[i];
        const int64_t v = item_vectors(it, L, lay);
        need[i] = std::max<int64_t>(1, cdiv(v, threads));
        weight[i] = std::max<int64_t>(1, v) * (it.in_cnt + (it.acc_rank >= 0 ? 1 : 0) + item_outputs(it));
        total += need[i];
        wsum += weight[i];
    }
    const int budget = std::max(max_ctas, ni);
    int begin = 0;
    for (int i = 0; i < ni; i++) {
        int64_t c = need[i];
        if (total > budget) c = std::min(need[i], std::max<int64_t>(1, weight[i] * budget / wsum));
        // at least one CTA per segment: the step kernel gives each of an
        // item's segments its own CTAs
        c = std::max<int64_t>(c, (int64_t)L.items[i].seg_width * L.items[i].seg_reps);
        L.items[i].cta_begin = begin;
        begin += (int)c;
    }
    return begin;
}

}  // namespace hc
