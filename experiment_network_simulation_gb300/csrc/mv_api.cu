// mv_api.cu -- host side of the C ABI declared in include/mv.h: descriptor
// validation, workspace layout in the caller's device buffer, upload, the
// set-up kernels, the megakernel launch and the result download.  Nothing
// here allocates device memory.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <numeric>
#include <tuple>
#include <new>
#include <vector>

#include "mv_device.cuh"
#include "../../include/mv.h"

using namespace mv;

namespace {

struct Region {
    u64 off = 0, bytes = 0;
};

// Largest shared-memory image of one experiment's dynamic state; larger
// experiments keep their state in global memory (wake table still staged).
constexpr u64 kStageMax = 112 * 1024;
// Shared-memory image budget when some experiment does not fit whole: what
// is left for one of two blocks an SM after the per-warp scratch.
constexpr u32 kPartialImage = 88 * 1024;
// ... and for the build with one 16-warp block an SM
constexpr u32 kPartialImage3 = 192 * 1024;
// Largest dynamic shared memory of a block (227 KiB) less the kernel's own
// static shared memory, for the builds with one block an SM.
constexpr u32 kBlockSmem = 227 * 1024 - 3 * 1024;

// Byte layout of the workspace: a static part uploaded from the host, then
// a dynamic part cleared and filled by the set-up kernels.
struct Layout {
    // counts
    u32 T = 0, W = 0, E = 0;
    u64 nsw = 0, nports = 0, nhosts = 0, nranks = 0, nnodes = 0, nedges = 0, ncolls = 0,
        nmemb = 0, na2a = 0, na2a_in = 0;
    u64 route_bytes = 0, q_total = 0, slot_total = 0, plog_total = 0, eg_total = 0,
        rk_total = 0, pend_total = 0, act_total = 0, lane_total = 0, portc_total = 0,
        nd_total = 0, rec_total = 0, coll_total = 0, taken_total = 0, items = 0,
        lcc_total = 0, rcc_total = 0;
    u32 warps = 1, image = 16;      // megakernel block size and shared image budget
    u32 variant = 1;                // 1: every experiment staged whole; 2: some are not
    u32 max_level = 0, max_nodes = 0, max_queues = 0, max_ranks = 0, max_colls = 0;
    u64 max_pairs = 0;
    // host copies of the derived tables
    std::vector<TopoRec> topo;
    std::vector<WorkRec> work;
    std::vector<ExpRec> exp;
    std::vector<u32> sw_pstart, port_sw, rank_first, succ_start, node_member, coll_mstart,
        memb_row, memb_col, node_rank, order;
    std::vector<uint2> sw_rec;
    std::vector<uint4> port_rec, host_rec;
    std::vector<CcRec> ccrec;
    // regions
    Region r_topo, r_work, r_exp, r_sw_nports, r_sw_level, r_sw_pstart, r_port_sw, r_port_peer,
        r_port_sigma, r_port_delta, r_host_port, r_host_sigma, r_host_delta, r_rank_first,
        r_rank_nnodes, r_node_kind, r_node_arg, r_node_npred, r_node_nsucc, r_succ_start,
        r_node_dur_lo, r_node_dur_hi, r_node_dur_key, r_succ, r_node_member, r_coll_kind,
        r_coll_intra, r_coll_nmembers, r_coll_parts, r_coll_alpha, r_coll_beta_num,
        r_coll_beta_den, r_coll_mstart, r_coll_bytes, r_member_rank, r_member_node,
        r_member_a2a_n, r_memb_row, r_a2a_dst, r_member_a2a_in_n, r_memb_col, r_a2a_in_src,
        r_a2a_bytes, r_a2a_in_bytes, r_mem, r_order, r_node_rank, r_sw_rec, r_port_rec,
        r_host_rec, r_ccrec;
    u64 static_bytes = 0;
    Region r_route, r_up_n, r_up_list, r_q_push, r_q_pop, r_q_taken, r_slots, r_eg, r_rk, r_rdirty, r_pend, r_act,
        r_lhot, r_lcold, r_ports, r_poplog, r_nd_pred, r_nd_cand, r_nd_start, r_nd_end, r_nd_pbase, r_nd_done,
        r_nd_out, r_ctl, r_rec_sender, r_rec_key, r_rec_tick, r_coll_start, r_coll_end, r_glob,
        r_wake, r_lcc, r_rcc;
    u64 total = 0;

    u64 cur = 0;
    Region take(u64 bytes)
    {
        Region r;
        r.off = cur;
        r.bytes = bytes;
        cur += (bytes + 255) / 256 * 256;
        return r;
    }
};

// Validate the descriptor and compute the layout.  Returns an MV_* code.
int plan(const mv_batch_desc *d, Layout &L)
{
    if (!d || d->version != 1 || d->n_topos == 0 || d->n_works == 0) return MV_EINVAL;
    L.T = d->n_topos;
    L.W = d->n_works;
    L.E = d->n_exps;
    // ---- topologies
    L.topo.resize(L.T);
    for (u32 t = 0; t < L.T; t++) {
        TopoRec &R = L.topo[t];
        R.nh = d->topo_nhosts[t];
        R.nsw = d->topo_nsw[t];
        R.nq = d->topo_nports[t];
        if (R.nh == 0 || R.nh > 65535 || R.nsw == 0) return MV_EINVAL;
        R.host_off = (u32)L.nhosts;
        R.sw_off = (u32)L.nsw;
        R.port_off = (u32)L.nports;
        R.route_off = L.route_bytes;
        R.rdv = kUnset;
        L.nhosts += R.nh;
        L.nsw += R.nsw;
        L.nports += R.nq;
        L.route_bytes += (u64)R.nsw * R.nh;
        L.max_pairs = std::max(L.max_pairs, (u64)R.nsw * R.nh);
        if (L.nports > 0xFFFFFFFFull || L.nsw > 0xFFFFFFFFull) return MV_EOVERFLOW;
    }
    L.sw_pstart.resize(L.nsw);
    L.port_sw.resize(L.nports);
    L.sw_rec.resize(L.nsw);
    L.port_rec.resize(L.nports);
    L.host_rec.resize(L.nhosts);
    for (u32 t = 0; t < L.T; t++) {
        TopoRec &R = L.topo[t];
        u32 q = 0;
        for (u32 s = 0; s < R.nsw; s++) {
            u32 np = d->sw_nports[R.sw_off + s], lev = d->sw_level[R.sw_off + s];
            if (np == 0 || np > kMaxPorts || lev == 0 || lev > 250 || np > R.nq - q)
                return MV_EINVAL;
            L.max_level = std::max(L.max_level, lev);
            R.maxlev = std::max(R.maxlev, lev);
            L.sw_pstart[R.sw_off + s] = q;
            for (u32 p = 0; p < np; p++) L.port_sw[R.port_off + q + p] = s;
            q += np;
        }
        if (q != R.nq) return MV_EINVAL;
        for (u32 p = 0; p < R.nq; p++) {
            i32 pe = d->port_peer[R.port_off + p];
            u32 sg = d->port_sigma[R.port_off + p], dl = d->port_delta[R.port_off + p];
            if (sg == 0 || sg > 65535 || dl >= kPopLog) return MV_EINVAL;
            R.rdv = std::min(R.rdv, dl + 1);
            if (pe >= 0) {
                if ((u32)pe >= R.nq || d->port_peer[R.port_off + pe] != (i32)p) return MV_EINVAL;
            } else {
                u32 h = (u32)(-(pe + 1));
                if (h >= R.nh || d->host_port[R.host_off + h] != p) return MV_EINVAL;
            }
        }
        for (u32 h = 0; h < R.nh; h++) {
            u32 hp = d->host_port[R.host_off + h];
            u32 sg = d->host_sigma[R.host_off + h], dl = d->host_delta[R.host_off + h];
            if (hp >= R.nq || d->port_peer[R.port_off + hp] != -(i32)(h + 1)) return MV_EINVAL;
            if (sg == 0 || sg > 65535 || dl >= kPopLog) return MV_EINVAL;
            R.rdv = std::min(R.rdv, dl + 1);
        }
        // packed records the forwarding and injection steps read per packet
        for (u32 s = 0; s < R.nsw; s++)
            L.sw_rec[R.sw_off + s] = make_uint2(L.sw_pstart[R.sw_off + s], d->sw_nports[R.sw_off + s]);
        for (u32 p = 0; p < R.nq; p++) {
            i32 pe = d->port_peer[R.port_off + p];
            u32 dq = pe >= 0 ? (u32)pe : R.nq + (u32)(-(pe + 1));
            u32 owner = pe >= 0 ? L.port_sw[R.port_off + pe] : (0x80000000u | (u32)(-(pe + 1)));
            L.port_rec[R.port_off + p] = make_uint4(dq, d->port_sigma[R.port_off + p],
                                                    d->port_delta[R.port_off + p], owner);
        }
        for (u32 h = 0; h < R.nh; h++) {
            u32 hp = d->host_port[R.host_off + h];
            L.host_rec[R.host_off + h] = make_uint4(hp, d->host_sigma[R.host_off + h],
                                                    d->host_delta[R.host_off + h],
                                                    L.port_sw[R.port_off + hp]);
        }
        // pop log: only the last (delta + 1) - 1 pops of a queue are ever read
        u32 dmax = 1;
        for (u32 p = 0; p < R.nq; p++) dmax = std::max(dmax, d->port_delta[R.port_off + p] + 1);
        for (u32 h = 0; h < R.nh; h++) dmax = std::max(dmax, d->host_delta[R.host_off + h] + 1);
        R.plog = 1;
        while (R.plog < dmax) R.plog *= 2;
    }
    // ---- workloads
    L.work.resize(L.W);
    for (u32 w = 0; w < L.W; w++) {
        WorkRec &R = L.work[w];
        R.nr = d->work_nranks[w];
        R.nn = d->work_nnodes[w];
        R.ncoll = d->work_ncolls[w];
        R.nmemb = d->work_nmembers[w];
        // a packet carries its sender's node in 25 bits, the top 256 values
        // reserved for control packets
        if (R.nn >= kCtlNode) return MV_EINVAL;
        R.rank_off = (u32)L.nranks;
        R.node_off = (u32)L.nnodes;
        R.edge_off = (u32)L.nedges;
        R.coll_off = (u32)L.ncolls;
        R.memb_off = (u32)L.nmemb;
        R.a2a_off = (u32)L.na2a;
        R.a2a_in_off = (u32)L.na2a_in;
        L.nranks += R.nr;
        L.nnodes += R.nn;
        L.nedges += d->work_nedges[w];
        L.ncolls += R.ncoll;
        L.nmemb += R.nmemb;
        L.na2a += d->work_na2a[w];
        L.na2a_in += d->work_na2a_in[w];
        if (L.nnodes > 0x7FFFFFFFull || L.nedges > 0xFFFFFFFFull || L.nmemb > 0xFFFFFFFFull ||
            L.na2a > 0xFFFFFFFFull || L.na2a_in > 0xFFFFFFFFull)
            return MV_EOVERFLOW;
    }
    L.rank_first.resize(L.nranks);
    L.succ_start.resize(L.nnodes);
    L.node_member.assign(L.nnodes, kUnset);
    L.node_rank.resize(L.nnodes);
    L.coll_mstart.resize(L.ncolls);
    L.memb_row.resize(L.nmemb);
    L.memb_col.resize(L.nmemb);
    std::vector<u32> node_rank;
    for (u32 w = 0; w < L.W; w++) {
        const WorkRec &R = L.work[w];
        node_rank.assign(R.nn, 0);
        u32 n = 0;
        for (u32 r = 0; r < R.nr; r++) {
            L.rank_first[R.rank_off + r] = n;
            u32 c = d->rank_nnodes[R.rank_off + r];
            if (c > R.nn - n) return MV_EINVAL;         // more nodes than the workload declares
            for (u32 k = 0; k < c; k++) {
                node_rank[n + k] = r;
                L.node_rank[R.node_off + n + k] = r;
            }
            n += c;
        }
        if (n != R.nn) return MV_EINVAL;
        u64 e = 0;
        for (u32 u = 0; u < R.nn; u++) {
            L.succ_start[R.node_off + u] = (u32)e;
            e += d->node_nsucc[R.node_off + u];
        }
        if (e != d->work_nedges[w]) return MV_EINVAL;
        for (u32 u = 0; u < R.nn; u++) {
            u32 k = d->node_kind[R.node_off + u];
            if (k > NODE_NET) return MV_EINVAL;
            if (k != NODE_COMPUTE && d->node_arg[R.node_off + u] >= R.ncoll) return MV_EINVAL;
            if (d->node_dur_hi[R.node_off + u] < d->node_dur_lo[R.node_off + u]) return MV_EINVAL;
            for (u32 j = 0; j < d->node_nsucc[R.node_off + u]; j++) {
                u32 v = d->succ[R.edge_off + L.succ_start[R.node_off + u] + j];
                if (v >= R.nn || node_rank[v] != node_rank[u]) return MV_EINVAL;
            }
        }
        std::vector<u32> indeg(R.nn, 0);
        for (u64 j = 0; j < d->work_nedges[w]; j++) indeg[d->succ[R.edge_off + j]]++;
        for (u32 u = 0; u < R.nn; u++)
            if (indeg[u] != d->node_npred[R.node_off + u]) return MV_EINVAL;
        u32 m = 0, ra = 0, ca = 0;
        for (u32 c = 0; c < R.ncoll; c++) {
            u32 g = R.coll_off + c, N = d->coll_nmembers[g], kind = d->coll_kind[g];
            L.coll_mstart[g] = m;
            if (N == 0 || N > 0xFFFF || kind > COLL_A2A) return MV_EINVAL;   // 16-bit member index
            if (d->coll_bytes[g] >= (1ull << 40)) return MV_EOVERFLOW;
            bool intra = d->coll_intra[g] != 0;
            if (intra && (d->coll_alpha[g] == 0 || d->coll_beta_den[g] == 0 ||
                          d->coll_beta_num[g] > (1u << 20)))
                return MV_EINVAL;
            if (!intra && kind == COLL_RELAY && d->coll_parts[g] == 0) return MV_EINVAL;
            if (!intra && kind == COLL_P2P && N != 2) return MV_EINVAL;
            if (N > R.nmemb - m) return MV_EINVAL;          // more members than declared
            for (u32 i = 0; i < N; i++) {
                u32 gm = R.memb_off + m + i;
                u32 rr = d->member_rank[gm], u = d->member_node[gm];
                if (rr >= R.nr || u >= R.nn || node_rank[u] != rr) return MV_EINVAL;
                u32 nk = d->node_kind[R.node_off + u];
                if (nk != (intra ? NODE_INTRA : NODE_NET) || d->node_arg[R.node_off + u] != c)
                    return MV_EINVAL;
                if (L.node_member[R.node_off + u] != kUnset) return MV_EINVAL;
                L.node_member[R.node_off + u] = i;
                L.memb_row[gm] = ra;
                L.memb_col[gm] = ca;
                if (d->member_a2a_n[gm] > d->work_na2a[w] - ra ||
                    d->member_a2a_in_n[gm] > d->work_na2a_in[w] - ca)
                    return MV_EINVAL;                       // more entries than declared
                for (u32 j = 0; j < d->member_a2a_n[gm]; j++) {
                    u32 dst = d->a2a_dst[R.a2a_off + ra + j];
                    if (dst >= N || dst == i || d->a2a_bytes[R.a2a_off + ra + j] >= (1ull << 40))
                        return MV_EINVAL;
                }
                for (u32 j = 0; j < d->member_a2a_in_n[gm]; j++)
                    if (d->a2a_in_src[R.a2a_in_off + ca + j] >= N) return MV_EINVAL;
                ra += d->member_a2a_n[gm];
                ca += d->member_a2a_in_n[gm];
            }
            m += N;
        }
        if (m != R.nmemb || ra != d->work_na2a[w] || ca != d->work_na2a_in[w]) return MV_EINVAL;
        for (u32 u = 0; u < R.nn; u++)
            if (d->node_kind[R.node_off + u] != NODE_COMPUTE &&
                L.node_member[R.node_off + u] == kUnset)
                return MV_EINVAL;
        const u64 *mm = d->mem + 10ull * w;
        if (mm[9] && (mm[1] == 0 || mm[2] == 0)) return MV_EINVAL;
    }
    // ---- experiments
    // Per-rank table strides: the fixed limit, or less when no rank of the
    // workload can ever need that many (each NET node adds at most its
    // channels x lanes-per-channel send lanes and that many receive
    // counters; first-fit placement never reaches past their sum), so that
    // results and overflow statuses are those of the fixed-size tables.
    struct Caps { u32 lane, port, pend, act; };
    std::map<std::tuple<u32, u32, u32>, Caps> caps_cache;
    auto caps_of = [&](u32 w, u32 nc, u32 algo) -> Caps {
        auto key = std::make_tuple(w, nc, algo);
        auto it = caps_cache.find(key);
        if (it != caps_cache.end()) return it->second;
        const WorkRec &R = L.work[w];
        Caps c = {1, 1, 1, 1};
        u32 n = 0;
        for (u32 r = 0; r < R.nr; r++) {
            u64 lanes = 0, ports = 0, acts = 0;
            u32 cnt = d->rank_nnodes[R.rank_off + r];
            for (u32 u = n; u < n + cnt; u++) {
                u32 k = d->node_kind[R.node_off + u];
                if (k == NODE_COMPUTE) continue;
                acts++;
                if (k != NODE_NET) continue;
                u32 kind = d->coll_kind[R.coll_off + d->node_arg[R.node_off + u]];
                bool one = kind == COLL_RELAY || kind == COLL_P2P;
                u64 per = (one ? 1ull : nc) * ((kind == COLL_AR && algo == ALGO_TREE) ? 3ull : 1ull);
                lanes += per;
                ports += (one || kind == COLL_A2A) ? 1ull : per;
            }
            c.lane = std::max<u32>(c.lane, (u32)std::min<u64>(lanes, kNLane));
            c.port = std::max<u32>(c.port, (u32)std::min<u64>(ports, kNPort));
            c.pend = std::max<u32>(c.pend, std::min<u32>(cnt, kNPend));
            c.act = std::max<u32>(c.act, (u32)std::min<u64>(acts, kNAct));
            n += cnt;
        }
        caps_cache[key] = c;
        return c;
    };
    // processing order: largest first (bytes moved over the network), so
    // the persistent blocks finish close together
    std::vector<u64> work_cost(L.W, 0);
    for (u32 w = 0; w < L.W; w++) {
        const WorkRec &R = L.work[w];
        for (u32 u = 0; u < R.nn; u++)
            if (d->node_kind[R.node_off + u] == NODE_NET)
                work_cost[w] += d->coll_bytes[R.coll_off + d->node_arg[R.node_off + u]] / 4096 + 1;
    }
    L.exp.resize(L.E);
    u64 items = 0;
    u32 max_items = 1;
    u64 full_max = 0, wake_max = 16;
    for (u32 e = 0; e < L.E; e++) {
        ExpRec &X = L.exp[e];
        std::memset(&X, 0, sizeof X);
        X.topo = d->exp_topo[e];
        X.work = d->exp_work[e];
        if (X.topo >= L.T || X.work >= L.W) return MV_EINVAL;
        const TopoRec &T = L.topo[X.topo];
        const WorkRec &W = L.work[X.work];
        X.algo = d->exp_algo[e];
        X.nc = d->exp_nc[e];
        X.chunk = d->exp_chunk[e];
        X.pkt = d->exp_pkt[e];
        X.cap = d->exp_cap[e];
        X.tick_ps = d->exp_tick_ps[e];
        X.rec_cap = d->exp_rec_cap[e];
        X.voq = d->exp_voq[e];
        X.dur_seed = d->exp_dur_seed[e];
        X.ecmp_seed = d->exp_ecmp_seed[e];
        X.gpu_mem = d->exp_gpu_mem[e];
        if (W.nr > T.nh || X.algo > ALGO_TREE || X.nc == 0 || X.nc > 1024 || X.pkt == 0 ||
            X.cap < 2 || X.cap > 1024 || X.tick_ps == 0 || X.voq > 1 || (X.voq && X.cap > 64))
            return MV_EINVAL;
        // with VOQs several packets can leave an ingress's buffer in one tick, so
        // its pop log keeps the last 64 pops (a whole buffer)
        X.plog = X.voq ? 64u : T.plog;
        // DCQCN parameters (n_exps records of MV_CC_FIELDS words; NULL: none)
        if (d->exp_cc) {
            const u32 *c = d->exp_cc + (u64)MV_CC_FIELDS * e;
            if (c[0] > kDctcp) return MV_EINVAL;
            if (c[0]) {
                CcRec R;
                std::memset(&R, 0, sizeof R);
                R.mode = c[0];
                R.kmin = c[1]; R.kmax = c[2]; R.pmax = c[3]; R.gshift = c[4]; R.n = c[5];
                R.k = c[6]; R.t = c[7]; R.b = c[8]; R.f = c[9]; R.rai = c[10]; R.rhai = c[11];
                R.rmin = c[12]; R.w0 = c[13]; R.wmax = c[14];
                if (R.mode == kDctcp &&
                    (X.voq || R.kmin != R.kmax || R.gshift == 0 || R.gshift > 16 || R.w0 == 0 ||
                     R.wmax < R.w0 || R.wmax > 65535))
                    return MV_EINVAL;
                if (R.mode == kDcqcn &&
                    (X.voq || R.kmin > R.kmax || R.pmax > 65536 || R.gshift == 0 || R.gshift > 16 ||
                     R.n == 0 || R.k == 0 || R.t == 0 || R.b == 0 || R.f > 65535 || R.rai > kLine ||
                     R.rhai > kLine || R.rmin == 0 || R.rmin > kLine))
                    return MV_EINVAL;
                L.ccrec.push_back(R);
                X.cc = (u32)L.ccrec.size();
            }
        }
        // chunk size matters for every kind but the relay
        if (X.chunk == 0) {
            for (u32 c = 0; c < W.ncoll; c++)
                if (!d->coll_intra[W.coll_off + c] && d->coll_kind[W.coll_off + c] != COLL_RELAY)
                    return MV_EINVAL;
        }
        Caps cp = caps_of(X.work, X.nc, X.algo);
        X.lane_cap = cp.lane;
        X.port_cap = cp.port;
        X.pend_cap = cp.pend;
        X.act_cap = cp.act;
        X.nq = T.nq + T.nh;
        X.nsw = T.nsw;
        X.nr = W.nr;
        X.nn = W.nn;
        X.q_off = L.q_total;
        X.slot_off = L.slot_total;
        X.plog_off = L.plog_total;
        X.eg_off = L.eg_total;
        X.rk_off = L.rk_total;
        X.pend_off = L.pend_total;
        X.act_off = L.act_total;
        X.lane_off = L.lane_total;
        X.portc_off = L.portc_total;
        X.nd_off = L.nd_total;
        X.rec_off = L.rec_total;
        X.coll_res_off = L.coll_total;
        X.taken_off = L.taken_total;
        X.lcc_off = L.lcc_total;
        X.rcc_off = L.rcc_total;
        L.q_total += X.nq;
        L.slot_total += (u64)X.nq * X.cap;
        L.plog_total += (u64)X.nq * X.plog;
        L.taken_total += X.voq ? T.nq : 0;
        L.lcc_total += X.cc ? (u64)W.nr * X.lane_cap : 0;
        L.rcc_total += X.cc ? W.nr : 0;
        L.eg_total += T.nq;
        L.rk_total += W.nr;
        L.pend_total += (u64)W.nr * X.pend_cap;
        L.act_total += (u64)W.nr * X.act_cap;
        L.lane_total += (u64)W.nr * X.lane_cap;
        L.portc_total += (u64)W.nr * X.port_cap;
        L.nd_total += W.nn;
        L.rec_total += X.rec_cap;
        L.coll_total += W.ncoll;
        L.max_colls = std::max(L.max_colls, W.ncoll);
        L.max_nodes = std::max(L.max_nodes, W.nn);
        L.max_queues = std::max(L.max_queues, X.nq);
        L.max_ranks = std::max(L.max_ranks, W.nr);
        X.item_off = (u32)items;
        X.n_items = T.nsw + (W.nr + 31) / 32;
        items += X.n_items;
        max_items = std::max(max_items, X.n_items);
        u64 off[IM_N];
        u64 img = image_layout(X, T, off);
        X.stage_bytes = img <= kStageMax ? (u32)img : 0;
        if (X.stage_bytes) full_max = std::max(full_max, img);
        wake_max = std::max(wake_max, im_round(12ull * X.n_items));
        if (L.nd_total > 0xFFFFFFFFull * 4 || items > 0xFFFFFFFFull) return MV_EOVERFLOW;
    }
    L.items = items;
    L.warps = std::min<u32>(8, max_items);
    // Build: 1 when every experiment fits in shared memory whole; else 2
    // (two 8-warp blocks an SM) when the hottest arrays of the largest
    // experiment fit its budget, 3 (one 16-warp block an SM, twice the
    // shared memory a block) when they do not.
    L.variant = 1;
    u64 hot_max = 0;
    for (u32 e = 0; e < L.E; e++) {
        const ExpRec &X = L.exp[e];
        if (X.stage_bytes) continue;
        L.variant = 2;
        u64 sz[IM_N];
        image_bytes(X, L.topo[X.topo], sz);
        u64 hot = 0;
        for (int k : {IM_WAKE, IM_SWREC, IM_UPN, IM_RDIRTY, IM_QPUSH, IM_QPOP, IM_HOSTREC, IM_EG,
                      IM_UPLIST})
            hot += im_round(sz[k]);
        hot_max = std::max(hot_max, hot);
    }
    if (L.variant == 2 && hot_max > kPartialImage) L.variant = 3;
    L.image = (u32)std::min<u64>(std::max(full_max, wake_max), kStageMax);
    // experiments that do not fit whole stage their hottest arrays in what
    // two blocks an SM leave of shared memory
    bool partial = false;
    for (u32 e = 0; e < L.E; e++) partial |= L.exp[e].stage_bytes == 0;
    if (partial) L.image = kPartialImage;      // build 2's budget; build 3 widens it
    L.order.resize(L.E);
    std::iota(L.order.begin(), L.order.end(), 0u);
    std::stable_sort(L.order.begin(), L.order.end(), [&](u32 a, u32 b) {
        return work_cost[L.exp[a].work] > work_cost[L.exp[b].work];
    });
    // ---- regions
    L.cur = 0;
    L.r_topo = L.take(sizeof(TopoRec) * L.T);
    L.r_work = L.take(sizeof(WorkRec) * L.W);
    L.r_exp = L.take(sizeof(ExpRec) * std::max<u32>(L.E, 1));
    L.r_sw_nports = L.take(4 * L.nsw);
    L.r_sw_level = L.take(4 * L.nsw);
    L.r_sw_pstart = L.take(4 * L.nsw);
    L.r_port_sw = L.take(4 * L.nports);
    L.r_port_peer = L.take(4 * L.nports);
    L.r_port_sigma = L.take(4 * L.nports);
    L.r_port_delta = L.take(4 * L.nports);
    L.r_host_port = L.take(4 * L.nhosts);
    L.r_host_sigma = L.take(4 * L.nhosts);
    L.r_host_delta = L.take(4 * L.nhosts);
    L.r_rank_first = L.take(4 * L.nranks);
    L.r_rank_nnodes = L.take(4 * L.nranks);
    L.r_node_kind = L.take(4 * L.nnodes);
    L.r_node_arg = L.take(4 * L.nnodes);
    L.r_node_npred = L.take(4 * L.nnodes);
    L.r_node_nsucc = L.take(4 * L.nnodes);
    L.r_succ_start = L.take(4 * L.nnodes);
    L.r_node_dur_lo = L.take(4 * L.nnodes);
    L.r_node_dur_hi = L.take(4 * L.nnodes);
    L.r_node_dur_key = L.take(4 * L.nnodes);
    L.r_succ = L.take(4 * L.nedges);
    L.r_node_member = L.take(4 * L.nnodes);
    L.r_coll_kind = L.take(4 * L.ncolls);
    L.r_coll_intra = L.take(4 * L.ncolls);
    L.r_coll_nmembers = L.take(4 * L.ncolls);
    L.r_coll_parts = L.take(4 * L.ncolls);
    L.r_coll_alpha = L.take(4 * L.ncolls);
    L.r_coll_beta_num = L.take(4 * L.ncolls);
    L.r_coll_beta_den = L.take(4 * L.ncolls);
    L.r_coll_mstart = L.take(4 * L.ncolls);
    L.r_coll_bytes = L.take(8 * L.ncolls);
    L.r_member_rank = L.take(4 * L.nmemb);
    L.r_member_node = L.take(4 * L.nmemb);
    L.r_member_a2a_n = L.take(4 * L.nmemb);
    L.r_memb_row = L.take(4 * L.nmemb);
    L.r_a2a_dst = L.take(4 * L.na2a);
    L.r_member_a2a_in_n = L.take(4 * L.nmemb);
    L.r_memb_col = L.take(4 * L.nmemb);
    L.r_a2a_in_src = L.take(4 * L.na2a_in);
    L.r_a2a_bytes = L.take(8 * L.na2a);
    L.r_a2a_in_bytes = L.take(8 * L.na2a_in);
    L.r_mem = L.take(80 * L.W);
    L.r_order = L.take(4ull * std::max<u32>(L.E, 1));
    L.r_sw_rec = L.take(8 * L.nsw);
    L.r_port_rec = L.take(16 * L.nports);
    L.r_host_rec = L.take(16 * L.nhosts);
    L.r_node_rank = L.take(4 * L.nnodes);
    L.r_ccrec = L.take(sizeof(CcRec) * L.ccrec.size());
    L.static_bytes = L.cur;
    L.r_route = L.take(L.route_bytes);
    L.r_up_n = L.take(L.nsw);
    L.r_up_list = L.take(L.nports);
    L.r_q_push = L.take(8 * L.q_total);
    L.r_q_pop = L.take(8 * L.q_total);
    L.r_q_taken = L.take(8 * L.taken_total);
    L.r_slots = L.take(16 * L.slot_total);
    L.r_eg = L.take(8 * L.eg_total);
    L.r_rk = L.take(sizeof(RankCtl) * L.rk_total);
    L.r_rdirty = L.take(4 * L.rk_total);
    L.r_pend = L.take(8ull * L.pend_total);
    L.r_act = L.take(4ull * L.act_total);
    L.r_lhot = L.take(sizeof(LaneHot) * L.lane_total);
    L.r_lcold = L.take(sizeof(LaneCold) * L.lane_total);
    L.r_ports = L.take(8ull * L.portc_total);
    L.r_poplog = L.take(4ull * L.plog_total);
    L.r_nd_pred = L.take(4 * L.nd_total);
    L.r_nd_cand = L.take(4 * L.nd_total);
    L.r_nd_start = L.take(4 * L.nd_total);
    L.r_nd_end = L.take(4 * L.nd_total);
    L.r_nd_pbase = L.take(4 * L.nd_total);
    L.r_nd_done = L.take(4 * L.nd_total);
    L.r_nd_out = L.take(4 * L.nd_total);
    L.r_ctl = L.take(sizeof(ExpCtl) * std::max<u32>(L.E, 1));
    L.r_rec_sender = L.take(4 * L.rec_total);
    L.r_rec_key = L.take(4 * L.rec_total);
    L.r_rec_tick = L.take(4 * L.rec_total);
    L.r_coll_start = L.take(4 * L.coll_total);
    L.r_coll_end = L.take(4 * L.coll_total);
    L.r_glob = L.take(sizeof(Glob));
    L.r_wake = L.take(12 * L.items);
    L.r_lcc = L.take(sizeof(LaneCC) * L.lcc_total);
    L.r_rcc = L.take(sizeof(RankCC) * L.rcc_total);
    L.total = L.cur;
    return MV_OK;
}

template <class T>
T *at(void *base, const Region &r)
{
    return reinterpret_cast<T *>(static_cast<char *>(base) + r.off);
}

Params make_params(void *ws, const Layout &L)
{
    Params P;
    std::memset(&P, 0, sizeof P);
    P.topo = at<TopoRec>(ws, L.r_topo);
    P.work = at<WorkRec>(ws, L.r_work);
    P.exp = at<ExpRec>(ws, L.r_exp);
    P.sw_nports = at<u32>(ws, L.r_sw_nports);
    P.sw_level = at<u32>(ws, L.r_sw_level);
    P.sw_pstart = at<u32>(ws, L.r_sw_pstart);
    P.port_sw = at<u32>(ws, L.r_port_sw);
    P.port_peer = at<i32>(ws, L.r_port_peer);
    P.port_sigma = at<u32>(ws, L.r_port_sigma);
    P.port_delta = at<u32>(ws, L.r_port_delta);
    P.host_port = at<u32>(ws, L.r_host_port);
    P.host_sigma = at<u32>(ws, L.r_host_sigma);
    P.host_delta = at<u32>(ws, L.r_host_delta);
    P.route = at<u8>(ws, L.r_route);
    P.up_n = at<u8>(ws, L.r_up_n);
    P.up_list = at<u8>(ws, L.r_up_list);
    P.rank_first = at<u32>(ws, L.r_rank_first);
    P.rank_nnodes = at<u32>(ws, L.r_rank_nnodes);
    P.node_kind = at<u32>(ws, L.r_node_kind);
    P.node_arg = at<u32>(ws, L.r_node_arg);
    P.node_npred = at<u32>(ws, L.r_node_npred);
    P.node_nsucc = at<u32>(ws, L.r_node_nsucc);
    P.succ_start = at<u32>(ws, L.r_succ_start);
    P.node_dur_lo = at<u32>(ws, L.r_node_dur_lo);
    P.node_dur_hi = at<u32>(ws, L.r_node_dur_hi);
    P.node_dur_key = at<u32>(ws, L.r_node_dur_key);
    P.succ = at<u32>(ws, L.r_succ);
    P.node_member = at<u32>(ws, L.r_node_member);
    P.coll_kind = at<u32>(ws, L.r_coll_kind);
    P.coll_intra = at<u32>(ws, L.r_coll_intra);
    P.coll_nmembers = at<u32>(ws, L.r_coll_nmembers);
    P.coll_parts = at<u32>(ws, L.r_coll_parts);
    P.coll_alpha = at<u32>(ws, L.r_coll_alpha);
    P.coll_beta_num = at<u32>(ws, L.r_coll_beta_num);
    P.coll_beta_den = at<u32>(ws, L.r_coll_beta_den);
    P.coll_mstart = at<u32>(ws, L.r_coll_mstart);
    P.coll_bytes = at<u64>(ws, L.r_coll_bytes);
    P.member_rank = at<u32>(ws, L.r_member_rank);
    P.member_node = at<u32>(ws, L.r_member_node);
    P.member_a2a_n = at<u32>(ws, L.r_member_a2a_n);
    P.memb_row = at<u32>(ws, L.r_memb_row);
    P.a2a_dst = at<u32>(ws, L.r_a2a_dst);
    P.member_a2a_in_n = at<u32>(ws, L.r_member_a2a_in_n);
    P.memb_col = at<u32>(ws, L.r_memb_col);
    P.a2a_in_src = at<u32>(ws, L.r_a2a_in_src);
    P.a2a_bytes = at<u64>(ws, L.r_a2a_bytes);
    P.a2a_in_bytes = at<u64>(ws, L.r_a2a_in_bytes);
    P.mem = at<u64>(ws, L.r_mem);
    P.q_push = at<u64>(ws, L.r_q_push);
    P.q_pop = at<u64>(ws, L.r_q_pop);
    P.q_taken = at<u64>(ws, L.r_q_taken);
    P.ccrec = at<CcRec>(ws, L.r_ccrec);
    P.lcc = at<LaneCC>(ws, L.r_lcc);
    P.rcc = at<RankCC>(ws, L.r_rcc);
    P.slots = at<uint4>(ws, L.r_slots);
    P.eg = at<uint2>(ws, L.r_eg);
    P.rk = at<RankCtl>(ws, L.r_rk);
    P.rdirty = at<u32>(ws, L.r_rdirty);
    P.pend = at<uint2>(ws, L.r_pend);
    P.act = at<u32>(ws, L.r_act);
    P.lhot = at<LaneHot>(ws, L.r_lhot);
    P.lcold = at<LaneCold>(ws, L.r_lcold);
    P.ports = at<uint2>(ws, L.r_ports);
    P.poplog = at<u32>(ws, L.r_poplog);
    P.nd_pred = at<u32>(ws, L.r_nd_pred);
    P.nd_cand = at<u32>(ws, L.r_nd_cand);
    P.nd_start = at<u32>(ws, L.r_nd_start);
    P.nd_end = at<u32>(ws, L.r_nd_end);
    P.nd_pbase = at<u32>(ws, L.r_nd_pbase);
    P.nd_done = at<u32>(ws, L.r_nd_done);
    P.nd_out = at<i32>(ws, L.r_nd_out);
    P.ctl = at<ExpCtl>(ws, L.r_ctl);
    P.rec_sender = at<u32>(ws, L.r_rec_sender);
    P.rec_key = at<u32>(ws, L.r_rec_key);
    P.rec_tick = at<u32>(ws, L.r_rec_tick);
    P.coll_start = at<u32>(ws, L.r_coll_start);
    P.coll_end = at<u32>(ws, L.r_coll_end);
    P.order = at<u32>(ws, L.r_order);
    P.sw_rec = at<uint2>(ws, L.r_sw_rec);
    P.port_rec = at<uint4>(ws, L.r_port_rec);
    P.host_rec = at<uint4>(ws, L.r_host_rec);
    P.node_rank = at<u32>(ws, L.r_node_rank);
    P.wake = at<u32>(ws, L.r_wake);
    P.n_exps = L.E;
    P.n_topos = L.T;
    P.glob = at<Glob>(ws, L.r_glob);
    P.watchdog_ns = 0;
    P.stage_limit = L.image;
    P.stage_mode = 0;
    return P;
}

void put(std::vector<char> &img, const Region &r, const void *src, u64 bytes)
{
    if (bytes) std::memcpy(img.data() + r.off, src, bytes);
}

}  // namespace

struct mv_ctx {
    Layout L;
    Params P;
    void *ws;
    cudaStream_t stream;
    std::vector<ExpCtl> host_ctl;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    bool timed = false;
};

namespace {
// dynamic state back to tick 0: clear, routing tables, per-experiment init
cudaError_t setup_dynamic(mv_ctx *c)
{
    const Layout &L = c->L;
    cudaError_t e = cudaMemsetAsync(static_cast<char *>(c->ws) + L.static_bytes, 0,
                                    L.total - L.static_bytes, c->stream);
    for (u32 lev = 1; lev <= L.max_level && e == cudaSuccess; lev++)
        e = launch_routes(c->P, L.max_pairs, lev, c->stream);
    if (e == cudaSuccess) e = launch_up_lists(c->P, (u32)L.nsw, c->stream);
    if (e == cudaSuccess && L.E)
        e = launch_init(c->P, L.max_nodes, L.max_queues, L.max_ranks, c->stream);
    return e;
}
}  // namespace

extern "C" {

const char *mv_strerror(int code)
{
    switch (code) {
    case MV_OK: return "ok";
    case MV_INCOMPLETE: return "tick budget reached; call mv_run again";
    case MV_EINVAL: return "invalid batch descriptor or argument";
    case MV_ENOMEM: return "workspace smaller than mv_workspace_bytes()";
    case MV_ECUDA: return "CUDA call failed";
    case MV_ETIMEOUT: return "run stopped by its watchdog; state kept at a tick boundary";
    case MV_EOVERFLOW: return "size or tick count beyond 32-bit limits";
    default: return "unknown status";
    }
}

int mv_workspace_bytes(const mv_batch_desc *desc, uint64_t *bytes)
{
    if (!bytes) return MV_EINVAL;
    Layout L;
    int rc = plan(desc, L);
    *bytes = rc == MV_OK ? L.total : 0;
    return rc;
}

int mv_result_sizes(const mv_batch_desc *desc, uint64_t *n_nodes, uint64_t *n_records,
                    uint64_t *n_colls)
{
    Layout L;
    int rc = plan(desc, L);
    if (rc != MV_OK) return rc;
    if (n_nodes) *n_nodes = L.nd_total;
    if (n_records) *n_records = L.rec_total;
    if (n_colls) *n_colls = L.coll_total;
    return MV_OK;
}

int mv_create(const mv_batch_desc *d, void *ws, uint64_t ws_bytes, void *stream, mv_ctx **out)
{
    if (!out || !ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MV_EINVAL;
    *out = nullptr;
    mv_ctx *c = new (std::nothrow) mv_ctx;
    if (!c) return MV_ENOMEM;
    int rc = plan(d, c->L);
    if (rc != MV_OK) { delete c; return rc; }
    Layout &L = c->L;
    if (ws_bytes < L.total) { delete c; return MV_ENOMEM; }
    c->ws = ws;
    c->stream = static_cast<cudaStream_t>(stream);
    c->P = make_params(ws, L);
    // static image
    std::vector<char> img(L.static_bytes, 0);
    put(img, L.r_topo, L.topo.data(), sizeof(TopoRec) * L.T);
    put(img, L.r_work, L.work.data(), sizeof(WorkRec) * L.W);
    put(img, L.r_exp, L.exp.data(), sizeof(ExpRec) * L.E);
    put(img, L.r_sw_nports, d->sw_nports, 4 * L.nsw);
    put(img, L.r_sw_level, d->sw_level, 4 * L.nsw);
    put(img, L.r_sw_pstart, L.sw_pstart.data(), 4 * L.nsw);
    put(img, L.r_port_sw, L.port_sw.data(), 4 * L.nports);
    put(img, L.r_port_peer, d->port_peer, 4 * L.nports);
    put(img, L.r_port_sigma, d->port_sigma, 4 * L.nports);
    put(img, L.r_port_delta, d->port_delta, 4 * L.nports);
    put(img, L.r_host_port, d->host_port, 4 * L.nhosts);
    put(img, L.r_host_sigma, d->host_sigma, 4 * L.nhosts);
    put(img, L.r_host_delta, d->host_delta, 4 * L.nhosts);
    put(img, L.r_rank_first, L.rank_first.data(), 4 * L.nranks);
    put(img, L.r_rank_nnodes, d->rank_nnodes, 4 * L.nranks);
    put(img, L.r_node_kind, d->node_kind, 4 * L.nnodes);
    put(img, L.r_node_arg, d->node_arg, 4 * L.nnodes);
    put(img, L.r_node_npred, d->node_npred, 4 * L.nnodes);
    put(img, L.r_node_nsucc, d->node_nsucc, 4 * L.nnodes);
    put(img, L.r_succ_start, L.succ_start.data(), 4 * L.nnodes);
    put(img, L.r_node_dur_lo, d->node_dur_lo, 4 * L.nnodes);
    put(img, L.r_node_dur_hi, d->node_dur_hi, 4 * L.nnodes);
    put(img, L.r_node_dur_key, d->node_dur_key, 4 * L.nnodes);
    put(img, L.r_succ, d->succ, 4 * L.nedges);
    put(img, L.r_node_member, L.node_member.data(), 4 * L.nnodes);
    put(img, L.r_coll_kind, d->coll_kind, 4 * L.ncolls);
    put(img, L.r_coll_intra, d->coll_intra, 4 * L.ncolls);
    put(img, L.r_coll_nmembers, d->coll_nmembers, 4 * L.ncolls);
    put(img, L.r_coll_parts, d->coll_parts, 4 * L.ncolls);
    put(img, L.r_coll_alpha, d->coll_alpha, 4 * L.ncolls);
    put(img, L.r_coll_beta_num, d->coll_beta_num, 4 * L.ncolls);
    put(img, L.r_coll_beta_den, d->coll_beta_den, 4 * L.ncolls);
    put(img, L.r_coll_mstart, L.coll_mstart.data(), 4 * L.ncolls);
    put(img, L.r_coll_bytes, d->coll_bytes, 8 * L.ncolls);
    put(img, L.r_member_rank, d->member_rank, 4 * L.nmemb);
    put(img, L.r_member_node, d->member_node, 4 * L.nmemb);
    put(img, L.r_member_a2a_n, d->member_a2a_n, 4 * L.nmemb);
    put(img, L.r_memb_row, L.memb_row.data(), 4 * L.nmemb);
    put(img, L.r_a2a_dst, d->a2a_dst, 4 * L.na2a);
    put(img, L.r_member_a2a_in_n, d->member_a2a_in_n, 4 * L.nmemb);
    put(img, L.r_memb_col, L.memb_col.data(), 4 * L.nmemb);
    put(img, L.r_a2a_in_src, d->a2a_in_src, 4 * L.na2a_in);
    put(img, L.r_a2a_bytes, d->a2a_bytes, 8 * L.na2a);
    put(img, L.r_a2a_in_bytes, d->a2a_in_bytes, 8 * L.na2a_in);
    put(img, L.r_mem, d->mem, 80 * L.W);
    put(img, L.r_order, L.order.data(), 4ull * L.E);
    put(img, L.r_ccrec, L.ccrec.data(), sizeof(CcRec) * L.ccrec.size());
    put(img, L.r_sw_rec, L.sw_rec.data(), 8 * L.nsw);
    put(img, L.r_port_rec, L.port_rec.data(), 16 * L.nports);
    put(img, L.r_host_rec, L.host_rec.data(), 16 * L.nhosts);
    put(img, L.r_node_rank, L.node_rank.data(), 4 * L.nnodes);
    cudaError_t e = cudaMemcpyAsync(ws, img.data(), L.static_bytes, cudaMemcpyHostToDevice,
                                    c->stream);
    if (e == cudaSuccess) e = setup_dynamic(c);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);   // img is freed on return
    if (e == cudaSuccess) e = cudaEventCreate(&c->ev0);
    if (e == cudaSuccess) e = cudaEventCreate(&c->ev1);
    if (e != cudaSuccess) {
        if (c->ev0) cudaEventDestroy(c->ev0);
        if (c->ev1) cudaEventDestroy(c->ev1);
        delete c;
        return MV_ECUDA;
    }
    c->host_ctl.resize(std::max<u32>(L.E, 1));
    *out = c;
    return MV_OK;
}

int mv_run_ex(mv_ctx *c, uint32_t max_ticks, const mv_run_opts *o, uint64_t *steps_done)
{
    if (!c) return MV_EINVAL;
    if (c->L.E == 0) return MV_OK;
    Params P = c->P;
    P.max_ticks = max_ticks;
    u32 warps = c->L.warps, grid = 0, variant = c->L.variant;
    if (o) {
        if (o->stage > 2 || o->variant > 4) return MV_EINVAL;
        P.watchdog_ns = o->watchdog_ns;
        P.stage_mode = o->stage;
        if (o->variant) variant = o->variant;
        if (o->block_warps) warps = o->block_warps;
        grid = o->grid_blocks;
    }
    const u32 max_warps = variant == 4 ? kMaxWarps : variant == 3 ? 16u : 8u;
    if (variant >= 3 && !(o && o->block_warps)) warps = max_warps;
    warps = std::min<u32>(warps, max_warps);
    // shared image budget: the batch's own (whole images) for the latency
    // build, else what the build's blocks an SM leave
    u32 image = c->L.image;
    if (variant == 2 && c->L.variant == 2) image = kPartialImage;
    if (variant == 3) image = std::max<u32>(c->L.image, kPartialImage3);
    if (variant == 4)
        image = std::max<u32>(c->L.image,
                              (kBlockSmem - warps * megakernel_scratch_bytes()) & ~15u);
    P.stage_limit = image;
    const u32 smem = megakernel_smem(warps, image);
    int bpsm = 0, nsm = 0;
    const bool cc = !c->L.ccrec.empty();     // the build with the DCQCN code
    cudaError_t e = megakernel_prepare(variant, cc, warps, smem, &bpsm, &nsm);
    if (e != cudaSuccess || bpsm == 0) return MV_ECUDA;
    u32 blocks = std::min<u32>(c->L.E, (u32)(bpsm * nsm));
    if (grid) blocks = std::min(blocks, grid);
    e = cudaMemsetAsync(P.glob, 0, sizeof(Glob), c->stream);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev0, c->stream);
    if (e == cudaSuccess) e = launch_megakernel(variant, cc, P, blocks, warps, smem, c->stream);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev1, c->stream);
    c->timed = e == cudaSuccess;
    Glob g;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&g, P.glob, sizeof g, cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(c->host_ctl.data(), P.ctl, sizeof(ExpCtl) * c->L.E,
                            cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return MV_ECUDA;
    if (steps_done) *steps_done = g.steps;
    if (g.error) return MV_ETIMEOUT;
    for (u32 i = 0; i < c->L.E; i++)
        if (c->host_ctl[i].status == EXP_RUNNING) return MV_INCOMPLETE;
    return MV_OK;
}

int mv_run(mv_ctx *c, uint32_t max_ticks, uint64_t *steps_done)
{
    return mv_run_ex(c, max_ticks, nullptr, steps_done);
}

int mv_results(mv_ctx *c, const mv_results_view *o)
{
    if (!c || !o) return MV_EINVAL;
    const Layout &L = c->L;
    cudaError_t e = cudaSuccess;
    if (L.E)
        e = cudaMemcpyAsync(c->host_ctl.data(), c->P.ctl, sizeof(ExpCtl) * L.E,
                            cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess && o->node_start && L.nd_total)
        e = cudaMemcpyAsync(o->node_start, c->P.nd_start, 4 * L.nd_total, cudaMemcpyDeviceToHost,
                            c->stream);
    if (e == cudaSuccess && o->node_end && L.nd_total)
        e = cudaMemcpyAsync(o->node_end, c->P.nd_end, 4 * L.nd_total, cudaMemcpyDeviceToHost,
                            c->stream);
    if (e == cudaSuccess && o->rec_sender && L.rec_total)
        e = cudaMemcpyAsync(o->rec_sender, c->P.rec_sender, 4 * L.rec_total,
                            cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess && o->rec_key && L.rec_total)
        e = cudaMemcpyAsync(o->rec_key, c->P.rec_key, 4 * L.rec_total, cudaMemcpyDeviceToHost,
                            c->stream);
    if (e == cudaSuccess && o->rec_tick && L.rec_total)
        e = cudaMemcpyAsync(o->rec_tick, c->P.rec_tick, 4 * L.rec_total, cudaMemcpyDeviceToHost,
                            c->stream);
    // per-collective times: reduced on the device from the per-node ticks
    if (e == cudaSuccess && (o->coll_start || o->coll_end) && L.coll_total) {
        e = launch_coll_times(c->P, L.max_colls, c->stream);
        if (e == cudaSuccess && o->coll_start)
            e = cudaMemcpyAsync(o->coll_start, c->P.coll_start, 4 * L.coll_total,
                                cudaMemcpyDeviceToHost, c->stream);
        if (e == cudaSuccess && o->coll_end)
            e = cudaMemcpyAsync(o->coll_end, c->P.coll_end, 4 * L.coll_total,
                                cudaMemcpyDeviceToHost, c->stream);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return MV_ECUDA;
    for (u32 i = 0; i < L.E; i++) {
        const ExpCtl &x = c->host_ctl[i];
        if (o->status) o->status[i] = x.status;
        if (o->now) o->now[i] = x.now;
        if (o->pkts_injected) o->pkts_injected[i] = x.pkts_injected;
        if (o->pkt_hops) o->pkt_hops[i] = x.pkt_hops;
        if (o->pkts_delivered) o->pkts_delivered[i] = x.pkts_delivered;
        if (o->msgs_delivered) o->msgs_delivered[i] = x.msgs_delivered;
        if (o->digest) o->digest[i] = x.digest;
        if (o->rec_count) o->rec_count[i] = x.rec_count;
    }
    if (o->end_tick)
        for (u32 i = 0; i < L.E; i++)
            o->end_tick[i] = c->host_ctl[i].end_max1 ? c->host_ctl[i].end_max1 - 1 : kUnset;
    return MV_OK;
}

int mv_reset(mv_ctx *c)
{
    if (!c) return MV_EINVAL;
    c->timed = false;
    return setup_dynamic(c) == cudaSuccess ? MV_OK : MV_ECUDA;
}

int mv_last_run_ms(mv_ctx *c, float *ms)
{
    if (!c || !ms || !c->timed) return MV_EINVAL;
    return cudaEventElapsedTime(ms, c->ev0, c->ev1) == cudaSuccess ? MV_OK : MV_ECUDA;
}

int mv_destroy(mv_ctx *c)
{
    if (!c) return MV_EINVAL;
    if (c->ev0) cudaEventDestroy(c->ev0);
    if (c->ev1) cudaEventDestroy(c->ev1);
    delete c;
    return MV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free one-shot entry point: same create/run/results/destroy path,
// with the workspace in this file-scope device array instead of caller memory.
static __device__ __align__(256) unsigned char g_static_scratch[MV_STATIC_SCRATCH_BYTES];
// Set-up token of the array's device copy: device data starts at zero when
// the module is (re)loaded on a device, so a token that no longer reads back
// means the cached address belongs to an earlier load (for example before a
// cudaDeviceReset) and the set-up runs again.
static __device__ unsigned long long g_static_token;

namespace {
constexpr int kStaticMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kStaticMaxDevices] = {};
unsigned long long g_static_tok[kStaticMaxDevices] = {};
unsigned long long g_static_next = 0;

// The array's device address for the current device: looked up (with that
// device current) by the first call on the device, and again whenever the
// module's device data was re-initialised since.  Host code cannot use the
// array's name as an address: it needs the device address.
int static_scratch(int dev, cudaStream_t st, void **out)
{
    std::lock_guard<std::mutex> lock(g_static_mu);
    unsigned long long tok = 0;
    if (g_static_ptr[dev]) {
        if (cudaMemcpyFromSymbolAsync(&tok, g_static_token, sizeof tok, 0,
                                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return MV_ECUDA;
    }
    if (!g_static_ptr[dev] || tok != g_static_tok[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MV_ECUDA;
        const unsigned long long t = ++g_static_next;
        if (cudaMemcpyToSymbolAsync(g_static_token, &t, sizeof t, 0, cudaMemcpyHostToDevice,
                                    st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return MV_ECUDA;
        g_static_ptr[dev] = p;
        g_static_tok[dev] = t;
    }
    *out = g_static_ptr[dev];
    return MV_OK;
}
}  // namespace

extern "C" int mv_simulate_static(const mv_batch_desc *desc, uint32_t max_ticks, void *stream,
                                  const mv_results_view *out, uint64_t *steps_done)
{
    if (!desc || !out) return MV_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) return MV_ECUDA;
    uint64_t need = 0;
    int rc = mv_workspace_bytes(desc, &need);
    if (rc != MV_OK) return rc;
    if (need > MV_STATIC_SCRATCH_BYTES) return MV_ENOMEM;
    void *scratch = nullptr;
    rc = static_scratch(dev, static_cast<cudaStream_t>(stream), &scratch);
    if (rc != MV_OK) return rc;
    mv_ctx *c = nullptr;
    rc = mv_create(desc, scratch, MV_STATIC_SCRATCH_BYTES, stream, &c);
    if (rc != MV_OK) return rc;
    int run = mv_run(c, max_ticks, steps_done);
    if (run >= 0) {
        int r2 = mv_results(c, out);
        if (r2 != MV_OK) run = r2;
    }
    mv_destroy(c);
    return run;
}
