// mv_kernel.cu -- the persistent sm_103a megakernel of the SPME packet
// simulator, plus its set-up kernels.
//
// One launch advances every experiment of the batch (Multiverse section 4.3:
// all systems fused in one kernel, launched once per batch).  Experiments
// are independent (section 5: nothing crosses experiments), so each one is
// stepped by one thread block: blocks of the persistent grid take
// experiments from a shared counter, largest first, and step them tick by
// tick with a block barrier as the per-tick synchronisation.  While a block
// holds an experiment, its whole state lives in shared memory when it fits;
// otherwise the hottest arrays that fit the build's budget do (wake table
// first) and the rest stays in global memory.
//
// Inside a block, work items are
//   - switches: plan + pull forwarding (section 4.2), two ports a lane, the
//     per-egress plan bitmaps in shared memory; the latency build forwards
//     one switch a warp pass, the others pack up to four (64 ports);
//   - groups of 32 ranks, a lane each: DAG advance with the analytic
//     intra-server model (sections 3.2, 4.1), NIC injection, NIC receive and
//     acknowledgements.
// Items are dealt to warps round-robin; a warp reads 32 of its wake ticks at
// once and ballots the items due at the current tick.  Three builds differ
// only in registers, warps and shared memory a block (k_megakernel<1..3>).  Reads of state another entity may
// change in the same tick see start-of-tick values: queue counters carry the
// tick of their last change (at most one push and one pop per queue and
// tick), start ticks are read as "joined before this tick", and completion
// counters are monotone with timestamped results.  That makes the parallel
// tick equal to the serial phase order, with a single barrier per tick.
#include "mv_device.cuh"

namespace mv {

constexpr u32 kFull = 0xffffffffu;

// ---------------------------------------------------------------- helpers
// splitmix64 finaliser (S. Vigna, splitmix64.c, public domain).
__device__ __forceinline__ u64 mix64(u64 z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}
__device__ __forceinline__ u64 cdiv(u64 a, u64 b) { return (a + b - 1) / b; }
// a / b and a mod b for a 32-bit divisor, in 32-bit arithmetic whenever the
// dividend fits (the usual case: message and chunk sizes), else in 64-bit
__device__ __forceinline__ u64 udiv(u64 a, u32 b)
{
    return (a >> 32) == 0 ? (u64)((u32)a / b) : a / b;
}
__device__ __forceinline__ u64 umod(u64 a, u32 b)
{
    return (a >> 32) == 0 ? (u64)((u32)a % b) : a % b;
}
// h mod n for 1 <= n <= 255 by Barrett reduction: with m = floor((2^64 - 1) / n),
// the estimate hi64(h * m) of floor(h / n) is low by at most two, so two
// conditional subtractions finish the remainder exactly.  m comes from a
// table the compiler fills; a 64-bit division per packet would cost far more.
struct BarrettTab {
    u64 m[256];
    constexpr BarrettTab() : m() { for (u32 n = 1; n < 256; n++) m[n] = ~0ull / n; }
};
__constant__ BarrettTab kBarrett = BarrettTab();
__device__ __forceinline__ u32 mod_small(u64 h, u32 n)
{
    u64 r = h - __umul64hi(h, kBarrett.m[n]) * n;
    if (r >= n) r -= n;
    if (r >= n) r -= n;
    return (u32)r;
}
// ring-buffer slot of counter x in a queue of cap slots (a mask when cap is
// a power of two, as in every configured batch)
__device__ __forceinline__ u32 slot_ix(u32 x, u32 cap)
{
    return (cap & (cap - 1)) == 0 ? (x & (cap - 1)) : x % cap;
}

// State shared between warps of the block may sit in shared or in global
// memory, so these accessors use generic addresses.  Volatile accesses keep
// the compiler from caching or splitting a word another warp may change in
// the same tick.
__device__ __forceinline__ u64 ld_vol64(const u64 *p) { return *reinterpret_cast<const volatile u64 *>(p); }
__device__ __forceinline__ void st_vol64(u64 *p, u64 v) { *reinterpret_cast<volatile u64 *>(p) = v; }
__device__ __forceinline__ u32 ld_vol32(const u32 *p) { return *reinterpret_cast<const volatile u32 *>(p); }
__device__ __forceinline__ void st_vol32(u32 *p, u32 v) { *reinterpret_cast<volatile u32 *>(p) = v; }
__device__ __forceinline__ u64 globaltimer()
{
    u64 t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- set-up
// Shortest up/down routing: a switch sends a packet down the lowest port
// under which its destination host sits, else up (ECMP over its up ports).
__global__ void k_routes(Params P, u32 level)
{
    for (u32 t = 0; t < P.n_topos; t++) {
        const TopoRec T = P.topo[t];
        u64 n = (u64)T.nsw * T.nh;
        for (u64 idx = blockIdx.x * (u64)blockDim.x + threadIdx.x; idx < n;
             idx += (u64)gridDim.x * blockDim.x) {
            u32 s = (u32)(idx / T.nh), d = (u32)(idx % T.nh);
            u32 gs = T.sw_off + s;
            if (P.sw_level[gs] != level) continue;
            u32 np = P.sw_nports[gs], p0 = P.sw_pstart[gs];
            u8 r = 0xFF;
            for (u32 p = 0; p < np && r == 0xFF; p++) {
                i32 pe = P.port_peer[T.port_off + p0 + p];
                if (pe < 0) {
                    if ((u32)(-pe - 1) == d) r = (u8)p;
                } else {
                    u32 s2 = P.port_sw[T.port_off + pe];
                    if (P.sw_level[T.sw_off + s2] < level &&
                        P.route[T.route_off + (u64)s2 * T.nh + d] != 0xFF)
                        r = (u8)p;
                }
            }
            P.route[T.route_off + idx] = r;
        }
    }
}

__global__ void k_up_lists(Params P)
{
    for (u32 t = 0; t < P.n_topos; t++) {
        const TopoRec T = P.topo[t];
        for (u32 s = blockIdx.x * blockDim.x + threadIdx.x; s < T.nsw; s += gridDim.x * blockDim.x) {
            u32 gs = T.sw_off + s, np = P.sw_nports[gs], p0 = P.sw_pstart[gs], k = 0;
            for (u32 p = 0; p < np; p++) {
                i32 pe = P.port_peer[T.port_off + p0 + p];
                if (pe >= 0 && P.sw_level[T.sw_off + P.port_sw[T.port_off + pe]] > P.sw_level[gs])
                    P.up_list[T.port_off + p0 + k++] = (u8)p;
            }
            P.up_n[gs] = (u8)k;
        }
    }
}

// GPU memory check before the run (Multiverse section 3.1).  The page gives
// no formula; read as 16 bytes per parameter (bf16 weights and gradients,
// fp32 Adam moments and master copy) over TP*PP, plus activations
// s*b*(34h + 5*a*s) bytes per layer (Korthikanti et al. 2022, an outside
// source) for min(m, PP) micro-batches in flight on a stage, over TP.
__device__ bool memory_fits(const u64 *m, u64 cap)
{
    if (m[9] == 0) return true;
    u64 weights = 16 * m[0] / (m[1] * m[2]);
    u64 per_layer = m[5] * m[6] * (34 * m[7] + 5 * m[8] * m[5]);
    u64 mm = m[4] < m[2] ? m[4] : m[2];
    u64 acts = m[3] * mm * per_layer / m[1];
    return weights + acts <= cap;
}

// Tick-0 state of experiment e; the block's x threads cover its entities.
__device__ void init_experiment(const Params &P, u32 e)
{
    const ExpRec X = P.exp[e];
    const WorkRec W = P.work[X.work];
    u32 i = blockIdx.x * blockDim.x + threadIdx.x;
    u32 stride = gridDim.x * blockDim.x;
    for (u32 u = i; u < X.nn; u += stride) {
        u64 g = X.nd_off + u;
        P.nd_pred[g] = P.node_npred[W.node_off + u];
        P.nd_start[g] = kUnset;
        P.nd_end[g] = kUnset;
    }
    for (u32 q = i; q < X.nq; q += stride) {
        P.q_push[X.q_off + q] = (u64)kUnset << 32;
        P.q_pop[X.q_off + q] = (u64)kUnset << 32;
    }
    // work items: switches wake on their first packet, rank groups at tick 0;
    // no pokes pending
    u32 *wk = P.wake + 3ull * X.item_off;
    for (u32 it = i; it < X.n_items; it += stride) {
        wk[it] = it < X.nsw ? kUnset : 0;
        wk[X.n_items + it] = kUnset;
        wk[2 * X.n_items + it] = kUnset;
    }
    bool fits = memory_fits(P.mem + 10 * (u64)X.work, X.gpu_mem);
    // roots (no predecessor) are scheduled at tick 0, in node order
    for (u32 r = i; r < X.nr; r += stride) {
        RankCtl c = {};
        u32 first = P.rank_first[W.rank_off + r], cnt = P.rank_nnodes[W.rank_off + r];
        bool over = false;
        for (u32 u = first; u < first + cnt && fits; u++) {
            if (P.node_npred[W.node_off + u] != 0) continue;
            if (c.npend == X.pend_cap) { over = true; break; }
            P.pend[X.pend_off + (u64)r * X.pend_cap + c.npend++] = make_uint2(u, 0);
        }
        c.pfirst = c.npend ? 0u : kUnset;
        P.rk[X.rk_off + r] = c;
        if (over) atomicCAS(&P.ctl[e].status, (u32)EXP_RUNNING, (u32)EXP_OVERFLOW);
    }
}

// blockIdx.y strides over experiments
__global__ void k_init(Params P)
{
    for (u32 e = blockIdx.y; e < P.n_exps; e += gridDim.y) init_experiment(P, e);
}

__global__ void k_init_ctl(Params P)
{
    for (u32 e = blockIdx.x * blockDim.x + threadIdx.x; e < P.n_exps; e += gridDim.x * blockDim.x) {
        const ExpRec X = P.exp[e];
        ExpCtl c = {};
        c.status = memory_fits(P.mem + 10 * (u64)X.work, X.gpu_mem) ? EXP_RUNNING : EXP_OOM;
        c.now = 0;
        c.nodes_left = X.nn;
        P.ctl[e] = c;
    }
}

// Per-collective times from the per-node ticks (Multiverse section 3.1: the
// system simulator learns of each flow's completion; a collective is done
// when its last member is): first member start, last member end, or kUnset
// while some member has not ended.  blockIdx.y strides over experiments,
// x threads over the workload's collectives.
__global__ void k_coll_times(Params P)
{
    for (u32 e = blockIdx.y; e < P.n_exps; e += gridDim.y) {
        const ExpRec &X = P.exp[e];
        const WorkRec W = P.work[X.work];
        for (u32 c = blockIdx.x * blockDim.x + threadIdx.x; c < W.ncoll; c += gridDim.x * blockDim.x) {
            const u32 g = W.coll_off + c, N = P.coll_nmembers[g];
            const u32 *mn = P.member_node + W.memb_off + P.coll_mstart[g];
            u32 lo = kUnset, hi = 0;
            for (u32 i = 0; i < N; i++) {
                const u64 u = X.nd_off + mn[i];
                lo = min(lo, P.nd_start[u]);
                hi = max(hi, P.nd_end[u]);       // kUnset (not ended) is the largest value
            }
            P.coll_start[X.coll_res_off + c] = lo;
            P.coll_end[X.coll_res_off + c] = hi;
        }
    }
}

// ---------------------------------------------------------------- block state
// The experiment a block holds: its records, and generic pointers to its
// slice of every dynamic array (shared memory when staged, global if not).
struct XV {
    ExpRec X;
    TopoRec T;
    WorkRec W;
    u32 e, staged, plog, pad;
    u64 *q_push, *q_pop, *q_taken;
    u32 *poplog;
    uint4 *slots;
    uint2 *eg;
    RankCtl *rk;
    u32 *rdirty;
    uint2 *pend;
    u32 *act;
    LaneHot *lhot;
    LaneCold *lcold;
    uint2 *ports;
    u32 *nd_pred, *nd_cand, *nd_start, *nd_end, *nd_pbase, *nd_done;
    i32 *nd_out;
    u32 *wake;
    const uint2 *sw_rec;
    const uint4 *port_rec, *host_rec;
    const u8 *route, *up_n, *up_list;
};

// The fields the per-tick code reads, copied from the block's view into
// registers at the start of each switch or rank-group step: stores through
// the state pointers (shared or global) cannot alias registers, so the
// compiler loads each field once.
struct HV {
    struct {
        u32 algo, nc, pkt, cap, tick_ps, rec_cap, nr, nsw, lane_cap, port_cap, pend_cap, act_cap, voq, cc;
        u64 chunk, dur_seed, ecmp_seed, rec_off, lcc_off, rcc_off;
    } X;
    struct { u32 nh, nq, rdv; } T;
    struct { u32 node_off, edge_off, coll_off, memb_off, a2a_off, a2a_in_off; } W;
    u32 plog;
    u64 *q_push, *q_pop, *q_taken;
    u32 *poplog;
    uint4 *slots;
    uint2 *eg;
    RankCtl *rk;
    u32 *rdirty;
    uint2 *pend;
    u32 *act;
    LaneHot *lhot;
    LaneCold *lcold;
    uint2 *ports;
    u32 *nd_pred, *nd_cand, *nd_start, *nd_end, *nd_pbase, *nd_done;
    i32 *nd_out;
    u32 *wake;
    const uint2 *sw_rec;
    const uint4 *port_rec, *host_rec;
    const u8 *route, *up_n, *up_list;
};

__device__ __forceinline__ HV make_hv(const XV &S)
{
    HV V;
    V.X.algo = S.X.algo; V.X.nc = S.X.nc; V.X.pkt = S.X.pkt; V.X.cap = S.X.cap;
    V.X.tick_ps = S.X.tick_ps; V.X.rec_cap = S.X.rec_cap; V.X.nr = S.X.nr; V.X.nsw = S.X.nsw;
    V.X.lane_cap = S.X.lane_cap; V.X.port_cap = S.X.port_cap; V.X.pend_cap = S.X.pend_cap;
    V.X.act_cap = S.X.act_cap; V.X.voq = S.X.voq; V.X.chunk = S.X.chunk; V.X.dur_seed = S.X.dur_seed;
    V.X.ecmp_seed = S.X.ecmp_seed; V.X.rec_off = S.X.rec_off;
    V.X.cc = S.X.cc; V.X.lcc_off = S.X.lcc_off; V.X.rcc_off = S.X.rcc_off;
    V.T.nh = S.T.nh; V.T.nq = S.T.nq; V.T.rdv = S.T.rdv;
    V.W.node_off = S.W.node_off; V.W.edge_off = S.W.edge_off; V.W.coll_off = S.W.coll_off;
    V.W.memb_off = S.W.memb_off; V.W.a2a_off = S.W.a2a_off; V.W.a2a_in_off = S.W.a2a_in_off;
    V.plog = S.plog;
    V.q_push = S.q_push; V.q_pop = S.q_pop; V.q_taken = S.q_taken; V.poplog = S.poplog; V.slots = S.slots; V.eg = S.eg;
    V.rk = S.rk; V.rdirty = S.rdirty; V.pend = S.pend; V.act = S.act; V.lhot = S.lhot; V.lcold = S.lcold;
    V.ports = S.ports;
    V.nd_pred = S.nd_pred; V.nd_cand = S.nd_cand; V.nd_start = S.nd_start; V.nd_end = S.nd_end;
    V.nd_pbase = S.nd_pbase; V.nd_done = S.nd_done; V.nd_out = S.nd_out; V.wake = S.wake;
    V.sw_rec = S.sw_rec; V.port_rec = S.port_rec; V.host_rec = S.host_rec; V.route = S.route;
    V.up_n = S.up_n; V.up_list = S.up_list;
    return V;
}

// How a step sees its experiment: a register copy (HV: fewest reloads, for
// the latency build) or the block's shared view itself (const XV &: fewest
// registers, for the occupancy build, whose state reads wait on HBM anyway).
template <class VT> struct ViewOf;
template <> struct ViewOf<HV> {
    __device__ __forceinline__ static HV get(const XV &s) { return make_hv(s); }
};
template <> struct ViewOf<const XV &> {
    __device__ __forceinline__ static const XV &get(const XV &s) { return s; }
};
template <class VT> struct kOnePerPass { static constexpr bool value = false; };
template <> struct kOnePerPass<HV> { static constexpr bool value = true; };
template <int VAR> struct ViewFor { typedef const XV &T; };
template <> struct ViewFor<1> { typedef HV T; };

// Per-experiment counters while a block holds it; only read after the last
// tick.  Decisions taken every tick use the per-warp reports instead, which
// are double-buffered so that one barrier per tick suffices.
struct Team {
    u32 end_max1, rec_count, now0, status0, left0, pad[3];
    unsigned long long pkts_injected, pkt_hops, pkts_delivered, msgs_delivered, digest;
    uint4 rep[2][kMaxWarps];    // per warp: (next wake, nodes completed, failure key, abort)
};

// Per-warp counters, kept in registers for the whole run of an experiment
// and added to the block's totals once at the end.
struct Acc {
    unsigned long long inj, hops, del, msg, dig;
    u32 emax;
};

// Failure keys: the lowest key of a tick wins, so rank failures (in rank
// order, as the serial phase order visits them) come before switch errors.
__device__ __forceinline__ u32 fail_key_rank(u32 r, u32 code) { return (r << 3) | code; }
constexpr u32 kFailSwitch = 0xF0000000u | EXP_ERROR;
constexpr u32 kFailReceive = 0xF1000000u;     // receive-phase failures order after the switches

// Per-warp scratch of one forwarding pass.  A pass handles a pack of up to
// kPack switches laid side by side over the 64 port positions (a lane has
// positions lane and lane + 32): switch k of the pack owns positions
// [base[k], base[k] + np[k]).
constexpr u32 kPack = 4;
struct SwSmem {
    uint4 pkt[kMaxPorts];
    unsigned long long mask[kMaxPorts];
    u32 head[kMaxPorts];
    u32 sw[kPack], base[kPack], np[kPack], p0[kPack], old[kPack], nxt[kPack];
};

// ---------------------------------------------------------------- credit
// Credit of queue qi for a sender at tick t: the queue holds `tail` pushes
// and `H` pops as of the start of the tick; the credit of a pop at tick x
// reaches the sender at x + D (D = delta + 1 of the link).  At most D - 1
// pops can still be on their way, so the pop log is only read when the
// queue is within D - 1 of full.
template <class VW>
__device__ __forceinline__ bool credit_ok(const VW &V, u32 qi, u32 tail, u32 H, u32 D, u32 t)
{
    const u32 cap = V.X.cap;
    if (tail - H + D - 1 < cap) return true;
    const u32 pm = V.plog - 1;
    const u32 *log = V.poplog + (u64)qi * V.plog;
    u32 back = 0;
    while (back < H && back + 1 < D) {
        if (ld_vol32(&log[(H - 1 - back) & pm]) + D <= t) break;
        back++;
    }
    return tail - (H - back) < cap;
}

// Credit of a switch ingress queue with virtual output queues: several of
// its packets may leave in one tick, so the sender reads the queue's current
// head (H pops so far, this tick's included) and walks back over its pop log
// (the last 64 pops: a whole buffer) until a pop whose credit has arrived.
// The consumer writes a pop's log entry before the head that announces it.
template <class VW>
__device__ __forceinline__ bool credit_ok_voq(const VW &V, u32 qi, u32 tail, u32 D, u32 t)
{
    const u32 H = (u32)ld_vol64(&V.q_pop[qi]);
    __threadfence_block();
    const u32 *log = V.poplog + (u64)qi * 64;
    u32 back = 0;
    while (back < H && back < 64) {
        if (ld_vol32(&log[(H - 1 - back) & 63u]) + D <= t) break;
        back++;
    }
    return tail - (H - back) < V.X.cap;
}

// ---------------------------------------------------------------- switches
template <class VW>
__device__ __forceinline__ u32 route_port(const VW &V, u32 s, u32 p0, uint4 pk)
{
    u8 r = V.route[(u64)s * V.T.nh + pk_dst(pk)];
    if (r != 0xFF) return r;
    u32 nup = V.up_n[s];
    if (nup == 0) return 0xFFu;
    u64 h = mix64((u64)pk_key(pk) ^ ((u64)s << 40) ^ V.X.ecmp_seed);
    return V.up_list[p0 + mod_small(h, nup)];
}

// ---------------------------------------------------------------- DCQCN
// Reaction point of a send lane (DCQCN, Zhu et al., SIGCOMM 2015; rates and
// alpha in units of 2^-20).  The state changes at notifications, at packets
// sent and at timer expiries; expiries are applied in time order whenever
// the lane's rate is about to be used, which is exact because nothing else
// reads it in between.
struct CcState {
    u32 rc, rt, alpha, next_tx, abase, rbase, tc, bc, sent;
};
__device__ __forceinline__ CcState cc_load(const LaneCC *p)
{
    const uint4 a = p->a, b = p->b;
    return CcState{a.x, a.y, a.z, a.w, b.x, b.y, b.z & 0xFFFFu, b.z >> 16, b.w};
}
__device__ __forceinline__ void cc_store(LaneCC *p, const CcState &S)
{
    p->a = make_uint4(S.rc, S.rt, S.alpha, S.next_tx);
    p->b = make_uint4(S.abase, S.rbase, S.tc | (S.bc << 16), S.sent);
}

// A rate increase event: fast recovery while both event counts are below F,
// hyper increase once both exceed it, additive increase otherwise; the
// current rate moves halfway to the target, rounded up.
__device__ __forceinline__ void cc_increase(const CcRec &C, CcState &S)
{
    const u32 mx = max(S.tc, S.bc), mn = min(S.tc, S.bc);
    u64 rt = S.rt;
    if (mx < C.f) {
    } else if (mn > C.f) {
        rt += (u64)(mn - C.f) * C.rhai;
    } else {
        rt += C.rai;
    }
    S.rt = rt > kLine ? kLine : (u32)rt;
    S.rc = (S.rt + S.rc + 1) / 2;
}

// Timer expiries up to tick t (alpha first on a tie): alpha decays every K
// ticks, the rate timer fires every T ticks.  Once neither can change
// anything but the timers' phase, the rest are counted in one step.  The
// loop runs at most (t - last expiry) / min(K, T) times.
__device__ __noinline__ void cc_catch_up(const CcRec &C, CcState &S, u32 t)
{
    for (;;) {
        if ((S.alpha >> C.gshift) == 0 && S.rc == kLine && S.rt == kLine) {
            if (t >= S.abase) S.abase += (t - S.abase) / C.k * C.k;
            if (t >= S.rbase) {
                const u32 n = (t - S.rbase) / C.t;
                S.rbase += n * C.t;
                S.tc = S.tc + n > 0xFFFFu ? 0xFFFFu : S.tc + n;
            }
            return;
        }
        const u64 ta = (u64)S.abase + C.k, tr = (u64)S.rbase + C.t;
        if (ta > t && tr > t) return;
        if (ta <= tr) {
            S.alpha -= S.alpha >> C.gshift;
            S.abase = (u32)ta;
        } else {
            S.rbase = (u32)tr;
            if (S.tc < 0xFFFFu) S.tc++;
            cc_increase(C, S);
        }
    }
}

// A notification taken at tick t: target = current rate, the current rate
// drops by alpha / 2 (not below Rmin), alpha moves toward 1 by g, the timers
// and the byte counter restart.
__device__ __noinline__ void cc_cut(const CcRec &C, CcState &S, u32 t)
{
    cc_catch_up(C, S, t);
    S.rt = S.rc;
    const u32 dec = (u32)(((u64)S.rc * S.alpha) >> 21);
    S.rc = S.rc - dec < C.rmin ? C.rmin : S.rc - dec;
    S.alpha = S.alpha - (S.alpha >> C.gshift) + (kLine >> C.gshift);
    if (S.alpha > kLine) S.alpha = kLine;
    S.abase = S.rbase = t;
    S.tc = S.bc = S.sent = 0;
}

// The lane sent a packet at tick t over an uplink of serialisation sigma.
__device__ __noinline__ void cc_sent(const CcRec &C, CcState &S, u32 sigma, u32 t)
{
    cc_catch_up(C, S, t);
    if (++S.sent >= C.b) {
        S.sent = 0;
        if (S.bc < 0xFFFFu) S.bc++;
        cc_increase(C, S);
    }
    S.next_tx = t + (u32)((((u64)sigma << 20) + S.rc - 1) / S.rc);
}

// Congestion point: a switch forwarding packet pk from ingress queue qin
// (of cap slots, counters h0..tl at the start of the tick) marks it by the
// number q of that queue's packets that had arrived by tick t (the packet
// included; those still on the wire do not count): never at q <= kmin,
// always above kmax, in between with probability pmax (q - kmin) / (kmax -
// kmin) drawn from a counter-based hash.  A queue's packets arrive in the
// order they were pushed, so q is found by bisection.
__device__ __noinline__ bool ecn_mark(const uint4 *slots, u32 cap, u64 seed, const CcRec &C,
                                      u32 qin, u32 h0, u32 tl, uint4 pk, u32 t)
{
    u32 lo = 0, hi = tl - h0;
    while (lo < hi) {
        const u32 mid = (lo + hi) / 2;
        if (slots[(u64)qin * cap + slot_ix(h0 + mid, cap)].x > t) hi = mid;
        else lo = mid + 1;
    }
    const u32 q = lo;
    if (q <= C.kmin) return false;
    if (q > C.kmax) return true;
    const u64 prob = (u64)C.pmax * (q - C.kmin) / (C.kmax - C.kmin);
    const u64 u = mix64(mix64(((u64)t << 32) | pk_key(pk)) ^ ((u64)qin << 40) ^ seed) & 0xFFFFu;
    return u < prob;
}

// Forwarding for one tick (Multiverse section 4.2) at the n switches of a
// pack (sm->sw/base/np/p0/old): each lane plans its ingress positions (the
// egress their ready head packet needs), then each lane pulls for its egress
// positions: free link, credit downstream, first planned ingress at or after
// the round-robin pointer.  Switches of a pack share nothing but the pass,
// so their steps are independent.  Pokes for other items go to `poke`.
// Returns the earliest tick this warp knows of at which something may happen
// (the switches' own next wakes and the wakes they gave other items); *fail
// gets a failure key.  `qstaged`: the queue words are in shared memory.
template <class VT>
__device__ __forceinline__ u32 switch_pack(const XV &Vs, Acc &acc, u32 n, u32 t, u32 *poke,
                                           SwSmem *sm, u32 *fail, bool qstaged)
{
    // the view (see ViewOf): as a register copy, stores through the state
    // pointers cannot alias it, so its fields are loaded once per tick
    VT V = ViewOf<VT>::get(Vs);
    const u32 lane = threadIdx.x & 31;
    const u32 cap = V.X.cap, pm = V.plog - 1;
    // segment bounds (warp-uniform): position p belongs to switch k when
    // base[k] <= p < base[k] + np[k]
    const u32 b1 = n > 1 ? sm->base[1] : 64u, b2 = n > 2 ? sm->base[2] : 64u,
              b3 = n > 3 ? sm->base[3] : 64u;
    const u32 end = sm->base[n - 1] + sm->np[n - 1];
    u32 seg_[2], lp_[2], np_[2], q_[2];
    u32 pk_min = kUnset;                // earliest tick poked into a downstream item
    bool bad = false;
    u32 tail_[2] = {0, 0}, head_[2] = {0, 0}, dhead_[2] = {0, 0}, dtail_[2] = {0, 0};
    uint2 st_[2] = {make_uint2(kUnset, 0), make_uint2(kUnset, 0)};
    uint4 pr_[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    uint4 pk_[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    // Issue the independent loads together: per position its ingress queue
    // words, its egress state and record, and (once the queue words are in)
    // the ingress head packet, so that the head packet and the port record
    // are in flight at the same time.  The head slot cannot change during
    // the tick: its upstream may only push into a slot freed before it.
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        const u32 p = lane + 32 * j;
        const u32 k = (p >= b1) + (p >= b2) + (p >= b3);
        seg_[j] = k;
        lp_[j] = p - sm->base[k];
        np_[j] = sm->np[k];
        q_[j] = sm->p0[k] + lp_[j];
        if (p >= end || lp_[j] >= np_[j]) { seg_[j] = kUnset; continue; }
        const u32 qi = q_[j];
        const u64 pw = ld_vol64(&V.q_push[qi]);
        tail_[j] = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
        head_[j] = (u32)V.q_pop[qi];
        st_[j] = V.eg[qi];
        pr_[j] = V.port_rec[qi];
        if (head_[j] != tail_[j]) pk_[j] = V.slots[(u64)qi * cap + slot_ix(head_[j], cap)];
    }
    // with the queue words in shared memory these are cheap, so every free
    // egress gets them now; in global memory only egresses that a packet
    // wants load them (below)
    if (qstaged) {
#pragma unroll
        for (u32 j = 0; j < 2; j++) {
            if (seg_[j] == kUnset || st_[j].x > t) continue;
            const u32 dq = pr_[j].x;
            const u64 dpop = ld_vol64(&V.q_pop[dq]);
            dhead_[j] = (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u);
            dtail_[j] = (u32)V.q_push[dq];
        }
    }
    sm->mask[lane] = 0;
    sm->mask[lane + 32] = 0;
    if (lane < kPack) sm->nxt[lane] = kUnset;
    __syncwarp();
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        const u32 p = lane + 32 * j, k = seg_[j];
        if (k == kUnset) continue;
        const u32 head = head_[j];
        sm->head[p] = head;
        if (head == tail_[j]) continue;
        const uint4 pk = pk_[j];
        if (pk.x > t) { atomicMin(&sm->nxt[k], pk.x); continue; }
        atomicMin(&sm->nxt[k], t + 1);  // a ready head: left or blocked, look again next tick
        const u32 tg = route_port(V, sm->sw[k], sm->p0[k], pk);
        if (tg >= np_[j]) { bad = true; continue; }
        sm->pkt[p] = pk;
        atomicOr(&sm->mask[sm->base[k] + tg], 1ull << p);
    }
    __syncwarp();
    u32 hops = 0;
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        const u32 p = lane + 32 * j, k = seg_[j];
        if (k == kUnset) continue;
        const unsigned long long M = sm->mask[p];
        if (!M) continue;
        const uint2 st = st_[j];
        if (st.x > t) continue;             // busy: its heads wake the switch at t+1
        const uint4 pr = pr_[j];            // downstream queue, sigma, delta, its owner
        const u32 dq = pr.x, sg = pr.y, dl = pr.z;
        if (!qstaged) {
            const u64 dpop = ld_vol64(&V.q_pop[dq]);
            dhead_[j] = (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u);
            dtail_[j] = (u32)V.q_push[dq];
        }
        const u32 dtail = dtail_[j];
        if (!credit_ok(V, dq, dtail, dhead_[j], dl + 1, t)) continue;
        const u32 base = sm->base[k], np = np_[j];
        const unsigned long long hi = M & (~0ull << (base + st.y));   // round robin from rr
        const u32 i = (u32)__ffsll((long long)(hi ? hi : M)) - 1;      // a position
        uint4 pk = sm->pkt[i];
        pk.x = t + sg + dl;
        pk.y += (dl + 1) << 16;
        V.slots[(u64)dq * cap + slot_ix(dtail, cap)] = pk;
        st_vol64(&V.q_push[dq], ((u64)t << 32) | (u32)(dtail + 1));
        V.eg[q_[j]] = make_uint2(t + sg, i - base + 1 == np ? 0u : i - base + 1);
        // pop the ingress this egress took (an ingress head wants one egress)
        const u32 qin = sm->p0[k] + (i - base), hd = sm->head[i];
        st_vol32(&V.poplog[(u64)qin * V.plog + (hd & pm)], t);
        st_vol64(&V.q_pop[qin], ((u64)t << 32) | (u32)(hd + 1));
        // the queue's owner: the peer switch, or the rank group of the host
        if (!(pr.w & 0x80000000u)) atomicMin(&poke[pr.w], pk.x);
        else if ((pr.w & 0x7FFFFFFFu) < V.X.nr) atomicMin(&poke[V.X.nsw + (pr.w & 0x7FFFFFFFu) / 32], pk.x);
        pk_min = min(pk_min, pk.x);
        hops++;
    }
    acc.hops += hops;                   // per lane; summed over the warp once per experiment
    if (__any_sync(kFull, bad)) *fail = min(*fail, kFailSwitch);
    __syncwarp();                       // sm->nxt complete
    u32 w = kUnset;
    if (lane < n) {                     // each switch's own next wake
        const u32 old = sm->old[lane];
        w = min(sm->nxt[lane], old > t ? old : kUnset);
        V.wake[sm->sw[lane]] = w;
    }
    const u32 r = __reduce_min_sync(kFull, min(w, pk_min));
    __syncwarp();
    return r;
}

// One switch for one tick (the latency build's form of switch_pack, with
// register reductions instead of the pack table).  Forwarding at switch s
// for one tick (Multiverse section 4.2): each lane
// plans its ingress ports (the egress their ready head packet needs), then
// each lane pulls for its egress ports: free link, credit downstream, first
// planned ingress at or after the round-robin pointer.  `old` is the
// switch's pending wake; pokes for other items go to `poke`.  Returns the
// earliest tick this warp knows of at which something may happen (its own
// next wake and the wakes it gave other items); *fail gets a failure key.
// `qstaged`: the queue words are in shared memory.
template <class VT>
__device__ __forceinline__ u32 switch_tick(const XV &Vs, Acc &acc, u32 s, u32 t, u32 old,
                                           u32 *poke, SwSmem *sm, u32 *fail, bool qstaged,
                                           const CcRec *ccr)
{
    // the view (see ViewOf): as a register copy, stores through the state
    // pointers cannot alias it, so its fields are loaded once per tick
    VT V = ViewOf<VT>::get(Vs);
    const u32 lane = threadIdx.x & 31;
    const uint2 sr = V.sw_rec[s];
    const u32 p0 = sr.x, np = sr.y;
    const u32 cap = V.X.cap, pm = V.plog - 1;
    u32 nxt = kUnset;                   // own next wake
    u32 pk_min = kUnset;                // earliest tick poked into a downstream item
    bool ready_any = false;
    bool bad = false;
    // Issue the independent loads together: per port (a lane has ports lane
    // and lane + 32) its ingress queue words, its egress state and record,
    // then the downstream queue words of each free egress.
    u32 tail_[2] = {0, 0}, head_[2] = {0, 0}, dhead_[2] = {0, 0}, dtail_[2] = {0, 0};
    uint2 st_[2] = {make_uint2(kUnset, 0), make_uint2(kUnset, 0)};
    uint4 pr_[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        const u32 p = lane + 32 * j;
        if (p >= np) continue;
        const u32 qi = p0 + p;
        const u64 pw = ld_vol64(&V.q_push[qi]);
        tail_[j] = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
        head_[j] = (u32)V.q_pop[qi];
        st_[j] = V.eg[qi];
        pr_[j] = V.port_rec[qi];
    }
    // with the queue words in shared memory these are cheap, so every free
    // egress gets them now; in global memory only egresses that a packet
    // wants load them (below)
    if (qstaged) {
#pragma unroll
        for (u32 j = 0; j < 2; j++) {
            if (lane + 32 * j >= np || st_[j].x > t) continue;
            const u32 dq = pr_[j].x;
            const u64 dpop = ld_vol64(&V.q_pop[dq]);
            dhead_[j] = (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u);
            dtail_[j] = (u32)V.q_push[dq];
        }
    }
    sm->mask[lane] = 0;
    sm->mask[lane + 32] = 0;
    __syncwarp();
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        u32 p = lane + 32 * j;
        if (p >= np) continue;
        const u32 qi = p0 + p, head = head_[j];
        sm->head[p] = head;
        if (head == tail_[j]) continue;
        uint4 pk = V.slots[(u64)qi * cap + slot_ix(head, cap)];
        if (pk.x > t) { nxt = min(nxt, pk.x); continue; }
        ready_any = true;
        u32 tg = route_port(V, s, p0, pk);
        if (tg >= np) { bad = true; continue; }
        sm->pkt[p] = pk;
        atomicOr(&sm->mask[tg], 1ull << p);
    }
    __syncwarp();
    u32 hops = 0;
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        u32 eg = lane + 32 * j;
        if (eg >= np) continue;
        unsigned long long M = sm->mask[eg];
        if (!M) continue;
        const uint2 st = st_[j];
        if (st.x > t) continue;             // busy: its heads wake the switch at t+1
        const uint4 pr = pr_[j];            // downstream queue, sigma, delta, its owner
        const u32 dq = pr.x, sg = pr.y, dl = pr.z;
        if (!qstaged) {
            const u64 dpop = ld_vol64(&V.q_pop[dq]);
            dhead_[j] = (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u);
            dtail_[j] = (u32)V.q_push[dq];
        }
        const u32 dtail = dtail_[j];
        if (!credit_ok(V, dq, dtail, dhead_[j], dl + 1, t)) continue;
        unsigned long long hi = st.y < 64 ? (M & (~0ull << st.y)) : 0ull;
        u32 i = (u32)__ffsll((long long)(hi ? hi : M)) - 1;
        uint4 pk = sm->pkt[i];
        if (ccr && !pk_ecn(pk) && pk_node(pk) < kCtlNode) {
            // DCQCN marking by the ingress queue the packet leaves
            const u64 iw = ld_vol64(&V.q_push[p0 + i]);
            const u32 itl = (u32)iw - ((u32)(iw >> 32) == t ? 1u : 0u);
            if (ecn_mark(V.slots, cap, V.X.ecmp_seed, *ccr, p0 + i, sm->head[i], itl, pk, t))
                pk.z |= 1u << 31;
        }
        pk.x = t + sg + dl;
        pk.y += (dl + 1) << 16;
        V.slots[(u64)dq * cap + slot_ix(dtail, cap)] = pk;
        st_vol64(&V.q_push[dq], ((u64)t << 32) | (u32)(dtail + 1));
        V.eg[p0 + eg] = make_uint2(t + sg, i + 1 == np ? 0u : i + 1);
        // pop the ingress this egress took (an ingress head wants one egress)
        const u32 hd = sm->head[i];
        st_vol32(&V.poplog[(u64)(p0 + i) * V.plog + (hd & pm)], t);
        st_vol64(&V.q_pop[p0 + i], ((u64)t << 32) | (u32)(hd + 1));
        // the queue's owner: the peer switch, or the rank group of the host
        if (!(pr.w & 0x80000000u)) atomicMin(&poke[pr.w], pk.x);
        else if ((pr.w & 0x7FFFFFFFu) < V.X.nr) atomicMin(&poke[V.X.nsw + (pr.w & 0x7FFFFFFFu) / 32], pk.x);
        pk_min = min(pk_min, pk.x);
        hops++;
    }
    acc.hops += hops;                   // per lane; summed over the warp once per experiment
    nxt = __reduce_min_sync(kFull, ready_any ? t + 1 : nxt);   // heads left or blocked: next tick
    pk_min = __reduce_min_sync(kFull, pk_min);
    if (__any_sync(kFull, bad)) *fail = min(*fail, kFailSwitch);
    u32 w = min(nxt, old > t ? old : kUnset);
    if (lane == 0) V.wake[s] = w;
    __syncwarp();
    return min(w, pk_min);
}

// Forwarding for one tick at switch s with virtual output queues (the VOQ
// variant of Multiverse section 4.2): an ingress buffer holds one FIFO per
// egress.  Plan: each lane scans its ingress buffers in arrival order (up to
// the first packet not yet ready: a buffer's packets are ready in arrival
// order) and marks, per egress, the ingresses holding a ready packet for it.
// Pull: the egresses in index order (one lane at a time); a free egress with
// credit downstream takes, from the first marked ingress at or after its
// round-robin pointer that no lower egress served in this tick, its oldest
// packet for it.  A packet leaving from the middle of a buffer frees its slot
// once the buffer's head passes it (q_taken marks the slots already gone).
template <class VT>
__device__ __forceinline__ u32 switch_voq(const XV &Vs, Acc &acc, u32 s, u32 t, u32 old,
                                          u32 *poke, SwSmem *sm, u32 *fail)
{
    VT V = ViewOf<VT>::get(Vs);
    const u32 lane = threadIdx.x & 31;
    const uint2 sr = V.sw_rec[s];
    const u32 p0 = sr.x, np = sr.y, cap = V.X.cap, pm = V.plog - 1;
    u32 nxt = kUnset, pk_min = kUnset;
    bool ready_any = false, bad = false;
    sm->mask[lane] = 0;
    sm->mask[lane + 32] = 0;
    __syncwarp();
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        const u32 p = lane + 32 * j;
        if (p >= np) continue;
        const u32 qi = p0 + p;
        const u64 pw = ld_vol64(&V.q_push[qi]);
        const u32 tail0 = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
        const u64 tk = V.q_taken[qi];
        u64 seen = 0;                   // egresses this ingress already offers a packet
        u32 x = (u32)V.q_pop[qi];
        for (u32 n = 0; x != tail0 && n < cap; n++, x++) {  // a buffer holds at most cap
            const u32 sl = slot_ix(x, cap);
            if ((tk >> sl) & 1ull) continue;
            const uint4 pk = V.slots[(u64)qi * cap + sl];
            if (pk.x > t) { nxt = min(nxt, pk.x); break; }
            ready_any = true;
            const u32 e = route_port(V, s, p0, pk);
            if (e >= np) { bad = true; continue; }
            if (!((seen >> e) & 1ull)) {
                seen |= 1ull << e;
                atomicOr(&sm->mask[e], 1ull << p);
            }
        }
    }
    __syncwarp();
    u64 used = 0;                       // ingresses that sent a packet this tick
    u32 hops = 0;
    for (u32 e = 0; e < np; e++) {
        const unsigned long long M = sm->mask[e] & ~used;
        u32 took = kUnset;
        if (M && lane == (e & 31)) {
            const u32 qe = p0 + e;
            const uint2 st = V.eg[qe];
            if (st.x <= t) {
                const uint4 pr = V.port_rec[qe];    // downstream queue, sigma, delta, its owner
                const u32 dq = pr.x, sg = pr.y, dl = pr.z;
                const u32 dtail = (u32)V.q_push[dq];
                bool ok;
                if (dq < V.T.nq) {
                    ok = credit_ok_voq(V, dq, dtail, dl + 1, t);
                } else {                            // a NIC's receive queue: one pop a tick
                    const u64 dpop = ld_vol64(&V.q_pop[dq]);
                    ok = credit_ok(V, dq, dtail, (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u),
                                   dl + 1, t);
                }
                const unsigned long long hi = M & (~0ull << st.y);      // round robin from rr
                const u32 i = (u32)__ffsll((long long)(hi ? hi : M)) - 1;
                const u32 qin = p0 + i;
                u64 tk = V.q_taken[qin];
                const u32 h0 = (u32)V.q_pop[qin];
                // its oldest packet for e (the plan saw a ready one among the
                // buffer's cap slots)
                u32 x = h0, n = 0;
                uint4 pk = make_uint4(0, 0, 0, 0);
                if (ok) {
                    for (; n < cap; n++, x++) {
                        const u32 sl = slot_ix(x, cap);
                        if ((tk >> sl) & 1ull) continue;
                        pk = V.slots[(u64)qin * cap + sl];
                        if (route_port(V, s, p0, pk) == e) break;
                    }
                    if (n == cap) { bad = true; ok = false; }
                }
                if (ok) {
                    pk.x = t + sg + dl;
                    pk.y += (dl + 1) << 16;
                    V.slots[(u64)dq * cap + slot_ix(dtail, cap)] = pk;
                    st_vol64(&V.q_push[dq], ((u64)t << 32) | (u32)(dtail + 1));
                    V.eg[qe] = make_uint2(t + sg, i + 1 == np ? 0u : i + 1);
                    // the slot is gone; the head moves past the gone slots
                    tk |= 1ull << slot_ix(x, cap);
                    const u32 tl = (u32)V.q_push[qin];
                    u32 h = h0;
                    while (h != tl && ((tk >> slot_ix(h, cap)) & 1ull)) {
                        tk &= ~(1ull << slot_ix(h, cap));
                        st_vol32(&V.poplog[(u64)qin * V.plog + (h & pm)], t);
                        h++;
                    }
                    V.q_taken[qin] = tk;
                    if (h != h0) {
                        __threadfence_block();      // log entries before the head that counts them
                        st_vol64(&V.q_pop[qin], ((u64)t << 32) | h);
                    }
                    if (!(pr.w & 0x80000000u)) atomicMin(&poke[pr.w], pk.x);
                    else if ((pr.w & 0x7FFFFFFFu) < V.X.nr)
                        atomicMin(&poke[V.X.nsw + (pr.w & 0x7FFFFFFFu) / 32], pk.x);
                    pk_min = min(pk_min, pk.x);
                    hops++;
                    took = i;
                }
            }
        }
        took = __shfl_sync(kFull, took, e & 31);
        if (took != kUnset) used |= 1ull << took;
    }
    acc.hops += hops;
    nxt = __reduce_min_sync(kFull, ready_any ? t + 1 : nxt);   // ready packets: next tick
    pk_min = __reduce_min_sync(kFull, pk_min);
    if (__any_sync(kFull, bad)) *fail = min(*fail, kFailSwitch);
    const u32 w = min(nxt, old > t ? old : kUnset);
    if (lane == 0) V.wake[s] = w;
    __syncwarp();
    return min(w, pk_min);
}

// ---------------------------------------------------------------- ranks
// A rank's control word while its lane works on it.
struct RankReg {
    u32 busy, rr, npend, nact;
    u64 lane_mask;
    u64 port_lo, port_hi;   // receive counters in use: bits 0..63, 64..127
    u32 blocked;    // every send lane waits for a receive count (no scan needed)
    u32 nintra;     // running intra-server memberships (checked every tick)
    u32 pfirst;     // start tick of the first pending node (kUnset: none), so
                    // that a tick with nothing due reads no pending list
};
static_assert(sizeof(RankCtl) == 48, "RankCtl is three 16-byte words");
__device__ __forceinline__ RankReg load_ctl(const RankCtl *p)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    uint4 a = q[0], b = q[1], c = q[2];
    RankReg r;
    r.busy = a.x; r.rr = a.y; r.npend = a.z; r.nact = a.w;
    r.lane_mask = ((u64)b.y << 32) | b.x;
    r.port_lo = ((u64)b.w << 32) | b.z;
    r.port_hi = ((u64)c.y << 32) | c.x;
    r.blocked = c.z & 1u;
    r.nintra = c.z >> 1;
    r.pfirst = c.w;
    return r;
}
__device__ __forceinline__ void store_ctl(RankCtl *p, const RankReg &r)
{
    uint4 *q = reinterpret_cast<uint4 *>(p);
    q[0] = make_uint4(r.busy, r.rr, r.npend, r.nact);
    q[1] = make_uint4((u32)r.lane_mask, (u32)(r.lane_mask >> 32), (u32)r.port_lo,
                      (u32)(r.port_lo >> 32));
    q[2] = make_uint4((u32)r.port_hi, (u32)(r.port_hi >> 32), r.blocked | (r.nintra << 1),
                      r.pfirst);
}
// A send lane while its rank's lane works on it (the stored form, Lane,
// packs the small fields).
struct LaneReg {
    u32 node, member, chan, kind;       // membership node, member index, channel, tree role
    u32 coll, nmemb, ckind, mbase;      // its collective, members, kind, first member entry
    u32 m, nmsg, pkts_left, dst_member;
    u32 dst_port, dep_base, dep_mask, dep_need;
    u32 key, a2a_e, a2a_start, dnode;
    u32 drank, dslot, ok_dst, pbase;
};
static_assert(sizeof(LaneHot) == 32 && sizeof(LaneCold) == 32, "lane records are 32 bytes");
static_assert(kNPort <= 256 && kNLane <= 256, "ports and channels fit the packed lane fields");
// Word by word: the local LaneReg never has its address taken, so it stays
// in registers.  A lane's member count, member index and destination member
// fit 16 bits (collectives have at most 65,535 members), its destination
// rank 16 bits (hosts), its receive slot, destination port, dependency base
// and counter base 8 bits (at most 128 receive counters a rank), its
// channel 8 bits (at most 64 lanes a rank).
__device__ __forceinline__ LaneReg load_lane_hot(const LaneHot *p)
{
    const uint4 a = p->a, b = p->b;
    LaneReg L;
    L.node = a.x;
    L.key = a.y & 0xFFFFFFu; L.dep_mask = (a.y >> 24) & 7u; L.ok_dst = (a.y >> 27) & 1u;
    L.pkts_left = a.z;
    L.drank = a.w & 0xFFFFu; L.dslot = (a.w >> 16) & 0xFFu; L.dst_port = a.w >> 24;
    L.dep_need = b.x;
    L.dep_base = b.y & 0xFFu; L.pbase = (b.y >> 8) & 0xFFu; L.chan = (b.y >> 16) & 0xFFu;
    L.kind = b.y >> 24;
    L.dnode = b.z; L.m = b.w;
    return L;
}
__device__ __forceinline__ void load_lane_cold(const LaneCold *p, LaneReg &L)
{
    const uint4 a = p->a, b = p->b;
    L.coll = a.x; L.nmemb = a.y & 0xFFFFu; L.member = a.y >> 16; L.mbase = a.z; L.nmsg = a.w;
    L.dst_member = b.x & 0xFFFFu; L.ckind = b.x >> 16; L.a2a_e = b.y; L.a2a_start = b.z;
}
__device__ __forceinline__ void store_lane_hot(LaneHot *p, const LaneReg &L)
{
    p->a = make_uint4(L.node, L.key | (L.dep_mask << 24) | (L.ok_dst << 27), L.pkts_left,
                      L.drank | (L.dslot << 16) | (L.dst_port << 24));
    p->b = make_uint4(L.dep_need, L.dep_base | (L.pbase << 8) | (L.chan << 16) | (L.kind << 24),
                      L.dnode, L.m);
}
__device__ __forceinline__ void store_lane_cold(LaneCold *p, const LaneReg &L)
{
    p->a = make_uint4(L.coll, L.nmemb | (L.member << 16), L.mbase, L.nmsg);
    p->b = make_uint4(L.dst_member | (L.ckind << 16), L.a2a_e, L.a2a_start, 0u);
}

// Receive-counter occupancy bits, by value (no indexed array, so the rank's
// control word stays in registers).
__device__ __forceinline__ bool port_used(const RankReg &C, u32 p)
{
    return ((p < 64 ? C.port_lo >> p : C.port_hi >> (p - 64)) & 1ull) != 0;
}
__device__ __forceinline__ void port_set(RankReg &C, u32 p, bool on)
{
    const u64 bit = 1ull << (p & 63);
    if (p < 64) C.port_lo = on ? (C.port_lo | bit) : (C.port_lo & ~bit);
    else C.port_hi = on ? (C.port_hi | bit) : (C.port_hi & ~bit);
}

// Per-rank view used while processing one tick.  CC: the kernel build
// handles DCQCN experiments (without it the DCQCN code is compiled out).
template <class VT, bool CC>
struct RankViewT {
    static constexpr bool kCC = CC;
    const Params *P;
    VT V;            // the view: a register copy (HV) or the block's shared view (const XV &)
    Team *TC;
    u32 *poke;          // this step's poke words of the experiment's items
    u32 r, t;
    RankReg C;
    bool changed, fail_over, fail_err;
    bool fail_rx;       // a table overflowed in the receive phase (after the switches)
    u32 nxt;            // this rank's own next wake
    u32 pk_min;         // earliest wake poked into other items
    u32 n_inj, n_del, n_msg, n_done, end_max1;
    u32 n_cnp;          // DCQCN notifications sent (packet-hops, not packets injected)
    u64 dig;
    __device__ __forceinline__ RankViewT(const Params *p, VT vv) : P(p), V(vv) {}
};

template <class RV>
__device__ __forceinline__ const auto &W_(const RV &v) { return v.V.W; }
template <class RV>
__device__ __forceinline__ const auto &X_(const RV &v) { return v.V.X; }
template <class RV>
__device__ __forceinline__ u32 coll_of(const RV &v, u32 u) { return v.P->node_arg[W_(v).node_off + u]; }
template <class RV>
__device__ __forceinline__ u32 nmemb(const RV &v, u32 c) { return v.P->coll_nmembers[W_(v).coll_off + c]; }
template <class RV>
__device__ __forceinline__ u32 ckind(const RV &v, u32 c) { return v.P->coll_kind[W_(v).coll_off + c]; }
template <class RV>
__device__ __forceinline__ u64 cbytes(const RV &v, u32 c) { return v.P->coll_bytes[W_(v).coll_off + c]; }
template <class RV>
__device__ __forceinline__ u32 mabs(const RV &v, u32 c, u32 i)
{
    return W_(v).memb_off + v.P->coll_mstart[W_(v).coll_off + c] + i;
}
template <class RV>
__device__ __forceinline__ u32 mrank(const RV &v, u32 c, u32 i) { return v.P->member_rank[mabs(v, c, i)]; }
template <class RV>
__device__ __forceinline__ u32 mnode(const RV &v, u32 c, u32 i) { return v.P->member_node[mabs(v, c, i)]; }
template <class RV>
__device__ __forceinline__ bool tree_of(const RV &v, u32 c)
{
    return ckind(v, c) == COLL_AR && X_(v).algo == ALGO_TREE;
}
template <class RV>
__device__ __forceinline__ u32 nchan(const RV &v, u32 c)
{
    u32 k = ckind(v, c);
    return (k == COLL_RELAY || k == COLL_P2P) ? 1u : X_(v).nc;
}
template <class RV>
__device__ __forceinline__ u32 nports_of(const RV &v, u32 c)
{
    u32 k = ckind(v, c);
    if (k == COLL_RELAY || k == COLL_P2P || k == COLL_A2A) return 1;
    return nchan(v, c) * (tree_of(v, c) ? 3u : 1u);
}
// channel c's share of S bytes (AutoCCL section 2.3: NC partitions)
__device__ __forceinline__ u64 part_bytes(u64 S, u32 nc, u32 c) { return S / nc + (c < S % nc ? 1 : 0); }
__device__ __forceinline__ u64 nchunks(u64 b, u64 C) { return b == 0 ? 1 : cdiv(b, C); }
template <class RV>
__device__ __forceinline__ u32 ring_steps(const RV &v, u32 c)
{
    u32 N = nmemb(v, c);
    if (N < 2) return 0;
    return ckind(v, c) == COLL_AR ? 2 * (N - 1) : N - 1;
}
template <class RV>
__device__ __forceinline__ u64 ring_loops(const RV &v, u32 c, u64 Pc)
{
    return Pc == 0 ? 1 : cdiv(Pc, (u64)nmemb(v, c) * X_(v).chunk);
}
template <class RV>
__device__ __forceinline__ u64 a2a_row_chunks(const RV &v, u32 c, u32 i)
{
    u32 m = mabs(v, c, i);
    u32 b = W_(v).a2a_off + v.P->memb_row[m], n = v.P->member_a2a_n[m];
    u64 tot = 0;
    for (u32 j = 0; j < n; j++) tot += nchunks(v.P->a2a_bytes[b + j], X_(v).chunk);
    return tot;
}

template <class RV>
__device__ __forceinline__ u32 lane_count(const RV &v, u32 c, u32 i, u32 ch, u32 kind)
{
    u32 N = nmemb(v, c);
    u64 S = cbytes(v, c);
    switch (ckind(v, c)) {
    case COLL_AR: case COLL_RS: case COLL_AG:
        if (tree_of(v, c)) {
            u64 n = nchunks(part_bytes(S, X_(v).nc, ch), X_(v).chunk);
            if (kind == 0) return i > 0 ? (u32)n : 0;
            return 2 * i + kind < N ? (u32)n : 0;
        }
        return (u32)(ring_loops(v, c, part_bytes(S, X_(v).nc, ch)) * ring_steps(v, c));
    case COLL_RELAY:
        return i + 1 < N ? v.P->coll_parts[W_(v).coll_off + c] : 0;
    case COLL_P2P:
        return i == 0 ? (u32)nchunks(S, X_(v).chunk) : 0;
    case COLL_A2A: {
        u64 tot = a2a_row_chunks(v, c, i);
        return tot > ch ? (u32)cdiv(tot - ch, X_(v).nc) : 0;
    }
    }
    return 0;
}

template <class RV>
__device__ __forceinline__ u32 port_count_expect(const RV &v, u32 c, u32 i, u32 p)
{
    u32 N = nmemb(v, c);
    u64 S = cbytes(v, c);
    switch (ckind(v, c)) {
    case COLL_AR: case COLL_RS: case COLL_AG:
        if (tree_of(v, c)) {
            u32 ch = p / 3, q = p % 3;
            u64 n = nchunks(part_bytes(S, X_(v).nc, ch), X_(v).chunk);
            if (q == 0) return i > 0 ? (u32)n : 0;
            return 2 * i + q < N ? (u32)n : 0;
        }
        return (u32)(ring_loops(v, c, part_bytes(S, X_(v).nc, p)) * ring_steps(v, c));
    case COLL_RELAY:
        return i > 0 ? v.P->coll_parts[W_(v).coll_off + c] : 0;
    case COLL_P2P:
        return i == 1 ? (u32)nchunks(S, X_(v).chunk) : 0;
    case COLL_A2A: {
        u32 m = mabs(v, c, i);
        u32 b = W_(v).a2a_in_off + v.P->memb_col[m], n = v.P->member_a2a_in_n[m];
        u64 tot = 0;
        for (u32 j = 0; j < n; j++) tot += nchunks(v.P->a2a_in_bytes[b + j], X_(v).chunk);
        return (u32)tot;
    }
    }
    return 0;
}

// Message L.m of a lane: bytes, destination member and port, and the own
// receive counts it waits for.  Returns its packet count.  The collective's
// member count, kind and first member entry come from the lane itself, so
// the only table reads are the collective's size and the destination's
// member entry, issued together.
template <class RV>
__device__ __forceinline__ u32 lane_setup(const RV &v, LaneReg &L)
{
    const Params &P = *v.P;
    const u32 c = L.coll, N = L.nmemb, i = L.member, m = L.m, ch = L.chan, nc = X_(v).nc;
    const u64 S = cbytes(v, c), C = X_(v).chunk;
    u64 bytes = 0;
    L.dep_mask = 0;
    L.dep_need = 0;
    L.dep_base = 0;
    switch (L.ckind) {
    case COLL_AR: case COLL_RS: case COLL_AG: {
        const u64 Pc = udiv(S, nc) + (ch < umod(S, nc) ? 1 : 0);    // channel ch's partition
        if (L.ckind == COLL_AR && X_(v).algo == ALGO_TREE) {
            bytes = Pc > (u64)m * C ? min(C, Pc - (u64)m * C) : 0;
            u32 kids = (2 * i + 1 < N ? 2u : 0u) | (2 * i + 2 < N ? 4u : 0u);
            if (L.kind == 0) {                        // reduce toward the root
                u32 par = (i - 1) / 2;
                L.dst_member = par;
                L.dst_port = ch * 3 + (i == 2 * par + 1 ? 1 : 2);
                L.dep_mask = kids;
            } else {                                  // broadcast to a child
                L.dst_member = 2 * i + L.kind;
                L.dst_port = ch * 3;
                L.dep_mask = i == 0 ? kids : 1u;
            }
            L.dep_need = m + 1;
            L.dep_base = ch * 3;
        } else {                                      // NCCL ring step order
            // a ring lane exists only for N >= 2, so steps >= 1
            const u32 steps = L.ckind == COLL_AR ? 2 * (N - 1) : N - 1;
            const u32 l = m / steps, kk = m - l * steps;
            const u64 stride = (u64)N * C;
            const u64 B = min(stride, Pc - (u64)l * stride);
            const u64 bs = udiv(B + N - 1, N);
            const u32 blk = (i + N - kk % N) % N;
            bytes = B > (u64)blk * bs ? min(bs, B - (u64)blk * bs) : 0;
            L.dst_member = (i + 1) % N;
            L.dst_port = ch;
            L.dep_base = ch;
            if (kk >= 1) { L.dep_mask = 1u; L.dep_need = l * steps + kk; }
        }
        break;
    }
    case COLL_RELAY: {                                // pipelined broadcast hop
        u32 K = P.coll_parts[W_(v).coll_off + c];
        bytes = udiv(S, K) + (m < umod(S, K) ? 1 : 0);
        L.dst_member = i + 1;
        L.dst_port = 0;
        if (i >= 1) { L.dep_mask = 1u; L.dep_need = m + 1; }
        break;
    }
    case COLL_P2P:
        bytes = S > (u64)m * C ? min(C, S - (u64)m * C) : 0;
        L.dst_member = 1;
        L.dst_port = 0;
        break;
    case COLL_A2A: {
        u32 mm = L.mbase + i;
        u32 r0 = W_(v).a2a_off + P.memb_row[mm];
        u64 g = (u64)ch + (u64)m * nc;
        while (g >= L.a2a_start + nchunks(P.a2a_bytes[r0 + L.a2a_e], C)) {
            L.a2a_start += (u32)nchunks(P.a2a_bytes[r0 + L.a2a_e], C);
            L.a2a_e++;
        }
        u64 j = g - L.a2a_start, b = P.a2a_bytes[r0 + L.a2a_e];
        bytes = b > j * C ? min(C, b - j * C) : 0;
        L.dst_member = P.a2a_dst[r0 + L.a2a_e];
        L.dst_port = 0;
        break;
    }
    }
    const u32 drank = P.member_rank[L.mbase + L.dst_member], dnode = P.member_node[L.mbase + L.dst_member];
    L.key = (u32)(mix64((u64)L.node | ((u64)(ch * 4 + L.kind) << 32) | ((u64)drank << 44)) &
                  0xFFFFFFu);
    if (dnode != L.dnode) {          // a new destination: its join is yet to be seen
        L.dnode = dnode;
        L.drank = drank;
        L.ok_dst = 0;
    }
    const u32 pkt = X_(v).pkt;
    return (u32)(bytes == 0 ? 1 : udiv(bytes + pkt - 1, pkt));
}

template <class RV>
__device__ __forceinline__ u32 compute_ticks(const RV &v, u32 u)
{
    const Params &P = *v.P;
    const u32 g = W_(v).node_off + u;
    u64 lo = P.node_dur_lo[g], hi = P.node_dur_hi[g], ns = lo;
    if (hi > lo) ns = lo + mix64(mix64((u64)P.node_dur_key[g]) ^ X_(v).dur_seed) % (hi - lo + 1);
    return (u32)cdiv(ns * 1000, X_(v).tick_ps);
}

// alpha + bytes/beta (Multiverse section 4.1), beta as ticks per byte
template <class RV>
__device__ __forceinline__ u32 intra_ticks(const RV &v, u32 c)
{
    const Params &P = *v.P;
    u32 cc = W_(v).coll_off + c;
    u64 g = nmemb(v, c), S = cbytes(v, c), be;
    switch (ckind(v, c)) {
    case COLL_AR: be = cdiv(2 * (g - 1) * S, g); break;
    case COLL_RS: case COLL_AG: be = cdiv((g - 1) * S, g); break;
    default: be = S;
    }
    return P.coll_alpha[cc] + (u32)cdiv(be * P.coll_beta_num[cc], P.coll_beta_den[cc]);
}

template <class VW>
__device__ __forceinline__ u32 rank_item(const VW &V, u32 r) { return V.X.nsw + r / 32; }

template <class RV>
__device__ __forceinline__ void rank_poke(RV &v, u32 item, u32 at)
{
    atomicMin(&v.poke[item], at);
    v.pk_min = min(v.pk_min, at);
}

// A member joined collective c at this tick: members waiting on its start
// look again when the join reaches them (intra-server barrier: next tick;
// network rendezvous: 1 + min(delta) ticks later).
template <class RV>
__device__ __forceinline__ void poke_members(RV &v, u32 c, u32 at)
{
    u32 N = nmemb(v, c), last = kUnset;
    for (u32 m = 0; m < N; m++) {
        u32 g = rank_item(v.V, mrank(v, c, m));
        if (g != last) rank_poke(v, g, at);
        last = g;
    }
}

// The pending list is kept sorted by (start tick, node): the nodes due at a
// tick are its prefix, already in node order.
template <class RV>
__device__ __forceinline__ void pend_add(RV &v, u32 u, u32 st)
{
    if (v.C.npend >= X_(v).pend_cap) { v.fail_over = true; return; }
    uint2 *pd = v.V.pend + (u64)v.r * X_(v).pend_cap;
    u32 j = v.C.npend++;
    while (j > 0) {
        const uint2 x = pd[j - 1];
        if (x.y < st || (x.y == st && x.x < u)) break;
        pd[j] = x;
        j--;
    }
    pd[j] = make_uint2(u, st);
    if (j == 0) v.C.pfirst = st;
}

template <class RV>
__device__ __forceinline__ void complete_node(RV &v, u32 u, u32 c)
{
    const Params &P = *v.P;
    const auto &V = v.V;
    V.nd_end[u] = c;
    v.n_done++;
    v.end_max1 = max(v.end_max1, c + 1);
    v.changed = true;
    if (c >= kTickLimit) { v.fail_over = true; return; }
    u32 s0 = P.succ_start[W_(v).node_off + u], ns = P.node_nsucc[W_(v).node_off + u];
    for (u32 j = 0; j < ns; j++) {
        u32 w = P.succ[W_(v).edge_off + s0 + j];
        u32 cd = max(V.nd_cand[w], c + 1);
        V.nd_cand[w] = cd;
        u32 left = V.nd_pred[w] - 1;
        V.nd_pred[w] = left;
        if (left == 0) pend_add(v, w, cd);
    }
}

template <class RV>
__device__ __forceinline__ void free_ports(RV &v, u32 u)
{
    u32 np = nports_of(v, coll_of(v, u)), b = v.V.nd_pbase[u];
    for (u32 p = b; p < b + np; p++) port_set(v.C, p, false);
}

// A rank joins a network collective: receive counters, then send lanes.
template <class RV>
__device__ __forceinline__ bool net_join(RV &v, u32 u)
{
    const Params &P = *v.P;
    const auto &V = v.V;
    const auto &X = V.X;
    u32 c = coll_of(v, u), i = P.node_member[W_(v).node_off + u];
    u32 np = nports_of(v, c);
    i32 base = -1;
    for (u32 b = 0; b + np <= X.port_cap && base < 0; b++) {
        u32 k = 0;
        while (k < np && !port_used(v.C, b + k)) k++;
        if (k == np) base = (i32)b;
    }
    if (base < 0) { v.fail_over = true; return false; }
    i32 out = 0;
    uint2 *ports = V.ports + (u64)v.r * X.port_cap;
    for (u32 p = 0; p < np; p++) {
        u32 s = (u32)base + p;
        port_set(v.C, s, true);
        ports[s] = make_uint2(0, u);
        out += (i32)port_count_expect(v, c, i, p);
    }
    u32 nch = nchan(v, c), lpc = tree_of(v, c) ? 3u : 1u;
    const u64 lane_ok = X.lane_cap >= 64 ? ~0ull : ((1ull << X.lane_cap) - 1);
    LaneHot *lhot = V.lhot + (u64)v.r * X.lane_cap;
    LaneCold *lcold = V.lcold + (u64)v.r * X.lane_cap;
    for (u32 ch = 0; ch < nch; ch++) {
        for (u32 kd = 0; kd < lpc; kd++) {
            u32 nm = lane_count(v, c, i, ch, kd);
            if (nm == 0) continue;
            u64 freem = ~v.C.lane_mask & lane_ok;
            if (!freem) { v.fail_over = true; return false; }
            u32 slot = (u32)__ffsll((long long)freem) - 1;
            LaneReg L = {};
            L.node = u; L.member = i; L.chan = ch; L.kind = kd;
            L.coll = c; L.nmemb = nmemb(v, c); L.ckind = ckind(v, c);
            L.mbase = W_(v).memb_off + P.coll_mstart[W_(v).coll_off + c];
            L.m = 0; L.nmsg = nm;
            L.dnode = kUnset;
            L.pbase = (u32)base;
            L.pkts_left = lane_setup(v, L);
            store_lane_hot(&lhot[slot], L);
            store_lane_cold(&lcold[slot], L);
            if (RV::kCC && X.cc) {
                LaneCC *lc = P.lcc + X.lcc_off + (u64)v.r * X.lane_cap + slot;
                const CcRec &C = P.ccrec[X.cc - 1];
                if (C.mode == kDctcp) {         // window w0, alpha = 1, first window: w0 packets
                    lc->a = make_uint4(C.w0 << 10, kLine, 0, 0);
                    lc->b = make_uint4(C.w0, 0, 0, 0);
                } else {                        // line rate, alpha = 1, timers from the join
                    cc_store(lc, CcState{kLine, kLine, kLine, 0, v.t, v.t, 0, 0, 0});
                }
            }
            v.C.lane_mask |= 1ull << slot;
            v.C.blocked = 0;
            out += (i32)nm;
        }
    }
    st_vol32(&V.nd_pbase[u], (u32)base);
    st_vol32(&V.nd_done[u], v.t);
    *reinterpret_cast<volatile i32 *>(&V.nd_out[u]) = out;
    return true;
}

// Running memberships in ascending node order; bit 31 marks an intra-server
// (analytic) one.
constexpr u32 kActIntra = 0x80000000u;
template <class RV>
__device__ __forceinline__ void act_add(RV &v, u32 u, u32 flag)
{
    if (v.C.nact >= X_(v).act_cap) { v.fail_over = true; return; }
    u32 *a = v.V.act + (u64)v.r * X_(v).act_cap;
    u32 j = v.C.nact;
    while (j > 0 && (a[j - 1] & ~kActIntra) > u) { a[j] = a[j - 1]; j--; }
    a[j] = u | flag;
    v.C.nact++;
    if (flag) v.C.nintra++;
}

// Schedule + AnalyticalSys: finish running memberships, then start the nodes
// scheduled for this tick (both in node order).
template <class RV>
__device__ __forceinline__ void dag_step(RV &v)
{
    const auto &V = v.V;
    const u32 t = v.t;
    uint2 *pd = V.pend + (u64)v.r * V.X.pend_cap;
    if (v.C.nact == 0 && v.C.pfirst > t) {      // nothing running or due
        v.nxt = min(v.nxt, v.C.pfirst);
        return;
    }
    // Running memberships: an intra-server one can finish whenever its last
    // member has started, so those are checked every tick; a network one
    // only once a membership of this rank has no message left (the receive
    // that takes its count to zero sets rdirty).
    u32 *a = V.act + (u64)v.r * V.X.act_cap;
    u32 w = 0;
    const bool dirty = ld_vol32(&V.rdirty[v.r]) != 0;
    if (dirty) atomicExch(&V.rdirty[v.r], 0u);
    const u32 nscan = (dirty || v.C.nintra) ? v.C.nact : 0;
    for (u32 j = 0; j < nscan; j++) {
        const u32 e = a[j], u = e & ~kActIntra;
        bool fin = false;
        if (e & kActIntra) {
            const u32 c = coll_of(v, u), N = nmemb(v, c);
            u32 b = 0;
            bool ok = true;
            for (u32 m = 0; m < N && ok; m++) {
                u32 st = ld_vol32(&V.nd_start[mnode(v, c, m)]);
                if (st == kUnset || st >= t) ok = false;
                else b = max(b, st);
            }
            if (ok) { complete_node(v, u, b + intra_ticks(v, c)); fin = true; v.C.nintra--; }
        } else if (ld_vol32((const u32 *)&V.nd_out[u]) == 0) {
            __threadfence_block();         // the count reached 0: read the latest event after it
            u32 done = ld_vol32(&V.nd_done[u]);
            free_ports(v, u);
            complete_node(v, u, done);
            fin = true;
        }
        if (!fin) { if (w != j) a[w] = e; w++; }
    }
    if (nscan) v.C.nact = w;
    // start the nodes due now: the prefix of the sorted pending list (a
    // start tick already past is an inconsistent schedule)
    if (v.C.pfirst < t) { v.fail_err = true; return; }
    u32 hi = 0;
    if (v.C.pfirst == t)
        while (hi < v.C.npend && pd[hi].y == t) hi++;
    for (u32 j = 0; j < hi && !v.fail_over; j++) {
        const u32 u = pd[j].x;
        v.changed = true;
        const u32 kind = v.P->node_kind[W_(v).node_off + u];
        if (kind == NODE_COMPUTE) {
            st_vol32(&V.nd_start[u], t);
            complete_node(v, u, t + compute_ticks(v, u));   // successors start later: after hi
        } else if (kind == NODE_INTRA) {
            st_vol32(&V.nd_start[u], t);
            act_add(v, u, kActIntra);
            poke_members(v, coll_of(v, u), t + 1);
        } else {
            if (!net_join(v, u)) break;
            st_vol32(&V.nd_start[u], t);
            poke_members(v, coll_of(v, u), t + V.T.rdv);
            if (ld_vol32((const u32 *)&V.nd_out[u]) == 0) {
                free_ports(v, u);
                complete_node(v, u, t);
            } else {
                act_add(v, u, 0);
            }
        }
    }
    if (v.fail_over || v.fail_err) return;
    // drop the started prefix; nodes scheduled above start later
    if (hi) {
        const u32 n = v.C.npend;
        u32 first = kUnset;
        for (u32 j = hi; j < n; j++) {
            const uint2 x = pd[j];
            if (j == hi) first = x.y;
            pd[j - hi] = x;
        }
        v.C.npend = n - hi;
        v.C.pfirst = first;
    }
    v.nxt = min(v.nxt, v.C.pfirst);
}

// SendSys + NICSndSys: one packet per uplink serialisation time, round-robin
// over the send lanes from the pointer; a lane is eligible once its receive
// dependencies are met and its destination joined before this tick.
// hr: the host's uplink record (queue, sigma, delta, switch); pw / tail:
// that queue's pop word and push count, loaded at the start of the tick.
template <class RV>
__device__ __forceinline__ void inject(RV &v, uint4 hr, u64 pw, u32 tail)
{
    const Params &P = *v.P;
    const auto &V = v.V;
    const auto &X = V.X;
    const u32 t = v.t;
    RankCC *rcc = (RV::kCC && X.cc) ? P.rcc + X.rcc_off + v.r : nullptr;
    const bool cnp = rcc && rcc->head != rcc->tail;     // control packets waiting
    const u32 ccmode = rcc ? P.ccrec[X.cc - 1].mode : 0u;
    if ((!v.C.lane_mask || v.C.blocked) && !cnp) return;
    if (v.C.busy > t) { v.nxt = min(v.nxt, v.C.busy); return; }
    const u32 qp = hr.x, hs = hr.y, hd = hr.z;
    u32 head = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
    if (!(X.voq ? credit_ok_voq(V, qp, tail, hd + 1, t) : credit_ok(V, qp, tail, head, hd + 1, t))) {
        v.nxt = min(v.nxt, t + 1);
        return;
    }
    if (cnp) {
        // a waiting notification goes first: one packet time, the lane
        // round-robin pointer stays
        const uint2 c = rcc->cq[rcc->head % kCtlRing];
        rcc->head++;
        uint4 pk;
        pk.x = t + hs + hd;
        pk.y = (c.x & 0xFFFFu) | ((hd + 1) << 16);
        pk.z = (kCtlNode + (c.x >> 22)) | (((c.x >> 16) & 63u) << 25);
        pk.w = c.y;
        V.slots[(u64)qp * X.cap + slot_ix(tail, X.cap)] = pk;
        st_vol64(&V.q_push[qp], ((u64)t << 32) | (u32)(tail + 1));
        v.C.busy = t + hs;
        v.n_cnp++;
        v.changed = true;
        rank_poke(v, hr.w, pk.x);
        if (v.C.lane_mask || rcc->head != rcc->tail) v.nxt = min(v.nxt, v.C.busy > t + 1 ? v.C.busy : t + 1);
        return;
    }
    u64 M = v.C.lane_mask;
    u64 hi = v.C.rr < 64 ? (M & (~0ull << v.C.rr)) : 0ull;
    u64 lo = M & ~hi;
    LaneHot *lhot = V.lhot + (u64)v.r * X.lane_cap;
    LaneCold *lcold = V.lcold + (u64)v.r * X.lane_cap;
    const uint2 *ports = V.ports + (u64)v.r * X.port_cap;
    bool timed = false;                 // some lane waits for a destination's join
    for (int pass = 0; pass < 2; pass++) {
        u64 m = pass == 0 ? hi : lo;
        while (m) {
            u32 l = (u32)__ffsll((long long)m) - 1;
            m &= m - 1;
            LaneReg L = load_lane_hot(&lhot[l]);    // all a packet needs
            LaneCC *lcc = nullptr;
            if (RV::kCC && ccmode) lcc = P.lcc + X.lcc_off + (u64)v.r * X.lane_cap + l;
            if (RV::kCC && ccmode == kDctcp && lcc->b.w) continue;   // all sent: waits for acks
            bool ok = true;
            for (u32 b = 0; b < 3 && ok; b++)
                if ((L.dep_mask >> b) & 1u)
                    if (ports[L.pbase + L.dep_base + b].x < L.dep_need) ok = false;
            if (!ok) continue;
            // receive counts only grow while the lane's message is current, so
            // a met dependency stays met: later packets of the message skip it
            // (the next message sets its own)
            L.dep_mask = 0;
            if (!L.ok_dst) {
                // the destination's join reaches this rank 1 + min(delta) ticks
                // later; when that time is known, it is this rank's own wake (a
                // poke alone could be shadowed by an earlier pending wake)
                const u32 dst_start = ld_vol32(&V.nd_start[L.dnode]);
                if (dst_start == kUnset) { timed = true; continue; }
                if (dst_start + V.T.rdv > t) {
                    v.nxt = min(v.nxt, dst_start + V.T.rdv);
                    timed = true;
                    continue;
                }
                L.dslot = ld_vol32(&V.nd_pbase[L.dnode]) + L.dst_port;
                L.ok_dst = 1;
            }
            CcState S;
            if (RV::kCC && ccmode == kDcqcn) {      // paced by its DCQCN rate
                S = cc_load(lcc);
                if (S.next_tx > t) {
                    v.nxt = min(v.nxt, S.next_tx);
                    timed = true;
                    continue;
                }
            }
            uint4 ca = make_uint4(0, 0, 0, 0);
            if (RV::kCC && ccmode == kDctcp) {      // its DCTCP window is full: waits for acks
                ca = lcc->a;
                if (ca.z - ca.w >= (ca.x >> 10)) continue;
            }
            uint4 pk;
            pk.x = t + hs + hd;
            pk.y = L.drank | ((hd + 1) << 16);
            pk.z = L.node | (l << 25);
            pk.w = L.key | ((L.pkts_left == 1 ? 1u : 0u) << 24) | (L.dslot << 25);
            V.slots[(u64)qp * X.cap + slot_ix(tail, X.cap)] = pk;
            st_vol64(&V.q_push[qp], ((u64)t << 32) | (u32)(tail + 1));
            v.C.busy = t + hs;
            v.C.rr = (l + 1) % kNLane;
            v.n_inj++;
            if (RV::kCC && ccmode == kDcqcn) {
                cc_sent(P.ccrec[X.cc - 1], S, hs, t);
                cc_store(lcc, S);
            }
            if (RV::kCC && ccmode == kDctcp) lcc->a.z = ca.z + 1;   // packets sent
            v.changed = true;
            rank_poke(v, hr.w, pk.x);
            if (--L.pkts_left == 0) {           // the message is out: the next one
                load_lane_cold(&lcold[l], L);
                if (++L.m == L.nmsg) {
                    // a DCTCP lane keeps its slot until every packet is acknowledged
                    if (RV::kCC && ccmode == kDctcp) lcc->b.w = 1;
                    else v.C.lane_mask &= ~(1ull << l);
                } else {
                    L.pkts_left = lane_setup(v, L);
                    store_lane_cold(&lcold[l], L);
                }
            }
            store_lane_hot(&lhot[l], L);
            if (v.C.lane_mask) v.nxt = min(v.nxt, v.C.busy > t + 1 ? v.C.busy : t + 1);
            return;
        }
    }
    // every lane waits for receive counts: nothing changes that but a
    // message completing at this rank (receive) or a new lane (join)
    if (!timed) v.C.blocked = 1;
}

// DCTCP sender (Alizadeh et al., SIGCOMM 2010): an acknowledgement of n
// packets, m of them marked, for lane l.  Once the packets sent before the
// last update are all acknowledged the observation window closes: alpha <-
// (1 - g) alpha + g F (F the marked fraction), and the window shrinks by
// alpha / 2 (not below one packet) if any was marked, else grows by one
// packet (up to wmax).  A draining lane frees its slot once every packet is
// acknowledged.
template <class RV>
__device__ __forceinline__ void dctcp_ack(RV &v, u32 l, u32 n, u32 m)
{
    const Params &P = *v.P;
    const auto &X = v.V.X;
    if (!((v.C.lane_mask >> l) & 1ull)) return;
    const CcRec &C = P.ccrec[X.cc - 1];
    LaneCC *lc = P.lcc + X.lcc_off + (u64)v.r * X.lane_cap + l;
    uint4 a = lc->a, b = lc->b;        // a: window, alpha, sent, acked; b: wend, wa, wm, draining
    a.w += n;
    b.y += n;
    b.z += m;
    if (a.w >= b.x) {
        const u32 F = (u32)(((u64)b.z << 20) / b.y);
        a.y = a.y - (a.y >> C.gshift) + (F >> C.gshift);
        if (b.z) {
            const u32 dec = (u32)(((u64)a.x * a.y) >> 21);
            a.x = a.x - dec < 1024u ? 1024u : a.x - dec;
        } else {
            a.x = min(a.x + 1024u, C.wmax << 10);
        }
        b.y = b.z = 0;
        b.x = a.z;
    }
    lc->a = a;
    lc->b = b;
    if (b.w && a.w == a.z) v.C.lane_mask &= ~(1ull << l);
}

// NICRcvSys + ACKSys: take the ready head of the downlink queue; the last
// packet of a message completes it at this rank and acknowledges it to the
// sender, sum over hops of (delta + 1) ticks later.
// ql / head / tail: the downlink queue and its start-of-tick counters; pk:
// its head packet (loaded at the start of the tick when the queue held one).
template <class RV>
__device__ __forceinline__ void receive(RV &v, u32 ql, u32 head, u32 tail, uint4 pk)
{
    const Params &P = *v.P;
    const auto &V = v.V;
    const auto &X = V.X;
    const u32 t = v.t;
    if (head == tail) return;
    if (pk.x > t) { v.nxt = min(v.nxt, pk.x); return; }
    st_vol32(&V.poplog[(u64)ql * V.plog + (head & (V.plog - 1))], t);
    st_vol64(&V.q_pop[ql], ((u64)t << 32) | (u32)(head + 1));
    v.changed = true;
    if (head + 1 != tail) v.nxt = min(v.nxt, t + 1);
    const u32 snd = pk_node(pk);
    if (RV::kCC && snd >= kCtlNode) {
        const u32 l = pk_lane(pk);
        if (P.ccrec[X.cc - 1].mode == kDctcp) {
            dctcp_ack(v, l, snd - kCtlNode, pk.w >> 24);
            v.C.blocked = 0;                   // its window may have room again:
            v.nxt = min(v.nxt, t + 1);         // the lanes look next tick
            return;
        }
        // DCQCN reaction point: the notification reaches the lane it names
        // if that lane still carries the flow
        if ((v.C.lane_mask >> l) & 1ull) {
            const LaneReg L = load_lane_hot(V.lhot + (u64)v.r * X.lane_cap + l);
            if (L.key == pk_key(pk)) {
                LaneCC *lcc = P.lcc + X.lcc_off + (u64)v.r * X.lane_cap + l;
                CcState S = cc_load(lcc);
                cc_cut(P.ccrec[X.cc - 1], S, t);
                cc_store(lcc, S);
            }
        }
        return;
    }
    v.n_del++;
    if (RV::kCC && X.cc && P.ccrec[X.cc - 1].mode == kDctcp) {
        // DCTCP: every data packet is acknowledged with its mark; the
        // newest acknowledgement still waiting for the same sender lane takes
        // it over (up to 255), else a new one joins the ring; a full ring is
        // a table overflow
        RankCC *rcc = P.rcc + X.rcc_off + v.r;
        const u32 id = P.node_rank[W_(v).node_off + snd] | (pk_lane(pk) << 16);
        const u32 mk = pk_ecn(pk);
        bool merged = false;
        for (u32 i = rcc->tail; i != rcc->head;) {      // at most kCtlRing entries
            uint2 &q = rcc->cq[--i % kCtlRing];
            if ((q.x & 0x3FFFFFu) != id) continue;
            if ((q.x >> 22) < 255u) {
                q.x += 1u << 22;
                q.y += mk << 24;
                merged = true;
            }
            break;
        }
        if (!merged) {
            if (rcc->tail - rcc->head >= kCtlRing) {
                v.fail_rx = true;
            } else {
                rcc->cq[rcc->tail % kCtlRing] = make_uint2(id | (1u << 22), pk_key(pk) | (mk << 24));
                rcc->tail++;
            }
        }
        v.nxt = min(v.nxt, t + 1);
    } else if (RV::kCC && pk_ecn(pk)) {
        // DCQCN notification point: at most one notification a flow per N
        // ticks (the last one per flow, direct-mapped by key); it waits in
        // this rank's ring (a full ring drops it) for the uplink
        RankCC *rcc = P.rcc + X.rcc_off + v.r;
        const u32 key = pk_key(pk), j = key % kNpTab;
        const uint2 e = rcc->np[j];
        const bool again = e.x == (key | 0x80000000u) &&
                           (u64)t < (u64)e.y + P.ccrec[X.cc - 1].n;
        if (!again && rcc->tail - rcc->head < kCnpRing) {
            rcc->np[j] = make_uint2(key | 0x80000000u, t);
            rcc->cq[rcc->tail % kCtlRing] =
                make_uint2(P.node_rank[W_(v).node_off + snd] | (pk_lane(pk) << 16), key);
            rcc->tail++;
            v.nxt = min(v.nxt, t + 1);
        }
    }
    if (!pk_last(pk)) return;
    v.nxt = min(v.nxt, t + 1);                         // DAG looks at its counts next tick
    uint2 *ports = V.ports + (u64)v.r * X.port_cap;
    u32 ps = pk_slot(pk);
    uint2 port = ports[ps];
    port.x++;
    ports[ps] = port;
    v.C.blocked = 0;
    u32 own = port.y;
    const u32 srank = P.node_rank[W_(v).node_off + snd];
    atomicMax(&V.nd_done[own], t);
    __threadfence_block();
    const i32 left_own = atomicSub(&V.nd_out[own], 1) - 1;
    atomicMax(&V.nd_done[snd], t + pk_hops(pk));
    __threadfence_block();
    const i32 left_snd = atomicSub(&V.nd_out[snd], 1) - 1;
    __threadfence_block();                 // counts before the flags that announce them
    // A membership can only finish when its count reaches zero, so only the
    // message that takes it there flags its rank for a look at its running
    // memberships (and, for the sender, wakes its rank group: the ACK).
    if (left_own == 0) atomicOr(&V.rdirty[v.r], 1u);
    if (left_snd == 0) {
        atomicOr(&V.rdirty[srank], 1u);
        rank_poke(v, rank_item(V, srank), t + 1);
    }
    v.n_msg++;
    v.dig += mix64(mix64((u64)snd | ((u64)pk_key(pk) << 32)) ^ (u64)t);
    u32 idx = atomicAdd(&v.TC->rec_count, 1u);
    if (idx < X.rec_cap) {
        P.rec_sender[X.rec_off + idx] = snd;
        P.rec_key[X.rec_off + idx] = pk_key(pk);
        P.rec_tick[X.rec_off + idx] = t;
    }
}

// Ranks g*32 .. g*32+31 for one tick, one lane each.  `old` is the group's
// pending wake; pokes for other items go to `poke`.  Returns the warp's
// earliest known next event; *done / *fail receive nodes completed and the
// failure key.
template <class VT, bool CC>
__device__ __forceinline__ u32 rank_tick(const Params &P, const XV &Vs, Team &TC, Acc &acc, u32 g,
                                         u32 t, u32 old, u32 *poke, u32 *done_out, u32 *fail)
{
    const u32 lane = threadIdx.x & 31;
    RankViewT<VT, CC> v(&P, ViewOf<VT>::get(Vs));     // the view (see ViewOf)
    v.TC = &TC;
    v.poke = poke;
    const auto &V = v.V;
    const u32 it = V.X.nsw + g;
    v.r = g * 32 + lane; v.t = t;
    v.changed = v.fail_over = v.fail_err = v.fail_rx = false;
    v.nxt = kUnset;
    v.pk_min = kUnset;
    v.n_inj = v.n_del = v.n_msg = v.n_done = v.end_max1 = v.n_cnp = 0;
    v.dig = 0;
    if (v.r < V.X.nr) {
        // issue the independent loads together: control word, uplink record,
        // downlink queue words; then the uplink queue words and the downlink
        // head packet
        v.C = load_ctl(&V.rk[v.r]);
        const uint4 hr = V.host_rec[v.r];
        const u32 ql = V.T.nq + v.r;
        const u64 rx_push = ld_vol64(&V.q_push[ql]);
        const u32 rx_head = (u32)V.q_pop[ql];
        const u32 rx_tail = (u32)rx_push - ((u32)(rx_push >> 32) == t ? 1u : 0u);
        const u64 up_pop = ld_vol64(&V.q_pop[hr.x]);
        const u32 up_tail = (u32)V.q_push[hr.x];
        uint4 rx_pk = make_uint4(kUnset, 0, 0, 0);
        if (rx_head != rx_tail) rx_pk = V.slots[(u64)ql * V.X.cap + slot_ix(rx_head, V.X.cap)];
        dag_step(v);
        if (!v.fail_over && !v.fail_err) {
            inject(v, hr, up_pop, up_tail);
            receive(v, ql, rx_head, rx_tail, rx_pk);
        }
        store_ctl(&V.rk[v.r], v.C);
    }
    const u32 nxt = __reduce_min_sync(kFull, v.nxt);
    const u32 pkm = __reduce_min_sync(kFull, v.pk_min);
    u32 done = 0;
    if (__any_sync(kFull, v.n_done != 0)) done = __reduce_add_sync(kFull, v.n_done);
    if (__any_sync(kFull, v.fail_over || v.fail_err || v.fail_rx)) {
        // failures in phase order: DAG step (by rank), switches, receive (by rank)
        u32 fk = v.fail_over ? fail_key_rank(v.r, EXP_OVERFLOW)
               : v.fail_err ? fail_key_rank(v.r, EXP_ERROR)
               : v.fail_rx ? kFailReceive | fail_key_rank(v.r, EXP_OVERFLOW) : kUnset;
        *fail = min(*fail, __reduce_min_sync(kFull, fk));
    }
    u32 w = min(nxt, old > t ? old : kUnset);
    if (lane == 0) V.wake[it] = w;
    // counters per lane; summed over the warp once per experiment
    acc.inj += v.n_inj;
    acc.hops += v.n_inj + v.n_cnp;
    acc.del += v.n_del;
    acc.msg += v.n_msg;
    acc.dig += v.dig;
    acc.emax = max(acc.emax, v.end_max1);
    *done_out += done;
    return min(w, pkm);
}

// ---------------------------------------------------------------- megakernel
// Copy n bytes between an experiment's global slice and its shared-memory
// image, all threads of the block (word copies when both sides allow).
__device__ __forceinline__ void block_copy(void *dst, const void *src, u64 n)
{
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | n) & 3) == 0) {
        u32 *d = reinterpret_cast<u32 *>(dst);
        const u32 *s = reinterpret_cast<const u32 *>(src);
        for (u64 i = threadIdx.x; i < n / 4; i += blockDim.x) d[i] = s[i];
    } else {
        u8 *d = reinterpret_cast<u8 *>(dst);
        const u8 *s = reinterpret_cast<const u8 *>(src);
        for (u64 i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
    }
}

// Global slice of array k of experiment X (k in the image order).
__device__ const void *global_slice(const Params &P, const ExpRec &X, const TopoRec &T, int k)
{
    switch (k) {
    case IM_WAKE: return P.wake + 3ull * X.item_off;
    case IM_QPUSH: return P.q_push + X.q_off;
    case IM_QPOP: return P.q_pop + X.q_off;
    case IM_EG: return P.eg + X.eg_off;
    case IM_RK: return P.rk + X.rk_off;
    case IM_RDIRTY: return P.rdirty + X.rk_off;
    case IM_PRED: return P.nd_pred + X.nd_off;
    case IM_CAND: return P.nd_cand + X.nd_off;
    case IM_START: return P.nd_start + X.nd_off;
    case IM_END: return P.nd_end + X.nd_off;
    case IM_PBASE: return P.nd_pbase + X.nd_off;
    case IM_DONE: return P.nd_done + X.nd_off;
    case IM_OUT: return P.nd_out + X.nd_off;
    case IM_ACT: return P.act + X.act_off;
    case IM_PEND: return P.pend + X.pend_off;
    case IM_PORTS: return P.ports + X.portc_off;
    case IM_POPLOG: return P.poplog + X.plog_off;
    case IM_LHOT: return P.lhot + X.lane_off;
    case IM_LCOLD: return P.lcold + X.lane_off;
    case IM_TAKEN: return P.q_taken + X.taken_off;
    case IM_SLOTS: return P.slots + X.slot_off;
    case IM_SWREC: return P.sw_rec + T.sw_off;
    case IM_PORTREC: return P.port_rec + T.port_off;
    case IM_HOSTREC: return P.host_rec + T.host_off;
    case IM_ROUTE: return P.route + T.route_off;
    case IM_UPN: return P.up_n + T.sw_off;
    default: return P.up_list + T.port_off;
    }
}

__device__ void set_slice(XV &V, int k, const void *c)
{
    void *p = const_cast<void *>(c);
    switch (k) {
    case IM_WAKE: V.wake = (u32 *)p; break;
    case IM_QPUSH: V.q_push = (u64 *)p; break;
    case IM_QPOP: V.q_pop = (u64 *)p; break;
    case IM_EG: V.eg = (uint2 *)p; break;
    case IM_RK: V.rk = (RankCtl *)p; break;
    case IM_RDIRTY: V.rdirty = (u32 *)p; break;
    case IM_PRED: V.nd_pred = (u32 *)p; break;
    case IM_CAND: V.nd_cand = (u32 *)p; break;
    case IM_START: V.nd_start = (u32 *)p; break;
    case IM_END: V.nd_end = (u32 *)p; break;
    case IM_PBASE: V.nd_pbase = (u32 *)p; break;
    case IM_DONE: V.nd_done = (u32 *)p; break;
    case IM_OUT: V.nd_out = (i32 *)p; break;
    case IM_ACT: V.act = (u32 *)p; break;
    case IM_PEND: V.pend = (uint2 *)p; break;
    case IM_PORTS: V.ports = (uint2 *)p; break;
    case IM_POPLOG: V.poplog = (u32 *)p; break;
    case IM_LHOT: V.lhot = (LaneHot *)p; break;
    case IM_LCOLD: V.lcold = (LaneCold *)p; break;
    case IM_TAKEN: V.q_taken = (u64 *)p; break;
    case IM_SLOTS: V.slots = (uint4 *)p; break;
    case IM_SWREC: V.sw_rec = (const uint2 *)p; break;
    case IM_PORTREC: V.port_rec = (const uint4 *)p; break;
    case IM_HOSTREC: V.host_rec = (const uint4 *)p; break;
    case IM_ROUTE: V.route = (const u8 *)p; break;
    case IM_UPN: V.up_n = (const u8 *)p; break;
    default: V.up_list = (const u8 *)p; break;
    }
}

// Arrays staged for an experiment that does not fit whole, most useful
// first: the per-item wake table, per-switch records, per-rank dirty words,
// the queue words, per-host records, egress state, the up lists.
__constant__ int kStagePrio[] = {IM_WAKE, IM_SWREC, IM_UPN, IM_RDIRTY, IM_QPUSH, IM_QPOP,
                                 IM_HOSTREC, IM_EG, IM_UPLIST, IM_RK, IM_PORTREC, IM_ACT};
constexpr int kNStagePrio = 12;

__shared__ XV s_V;
__shared__ Team s_TC;
__shared__ u64 s_off[IM_N];
__shared__ u64 s_sz[IM_N];
__shared__ u32 s_slot;

// Step experiment e from its clock until it finishes, stops, or reaches the
// run's tick budget; `img` is this block's shared-memory image space.
template <class VT, bool CC>
__device__ void run_experiment(const Params &P, u32 e, unsigned char *img, SwSmem *sm,
                               u64 t_start)
{
    XV &V = s_V;
    Team &TC = s_TC;
    const u32 warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nW = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        V.X = P.exp[e];
        V.T = P.topo[V.X.topo];
        V.W = P.work[V.X.work];
        V.e = e;
        V.plog = V.X.plog;
        const ExpCtl c = P.ctl[e];
        TC.end_max1 = c.end_max1;
        TC.rec_count = c.rec_count;
        TC.now0 = c.now;
        TC.status0 = c.status;
        TC.left0 = c.nodes_left;
        TC.pkts_injected = c.pkts_injected;
        TC.pkt_hops = c.pkt_hops;
        TC.pkts_delivered = c.pkts_delivered;
        TC.msgs_delivered = c.msgs_delivered;
        TC.digest = c.digest;
        image_bytes(V.X, V.T, s_sz);
        // What goes to shared memory: the whole image when it fits; else the
        // arrays of kStagePrio in that order while the budget lasts (mode 0),
        // the wake table alone (mode 1), or nothing (mode 2).
        u32 mask = 0;
        if (P.stage_mode == 0 && V.X.stage_bytes && V.X.stage_bytes <= P.stage_limit) {
            image_layout(V.X, V.T, s_off);
            mask = (1u << IM_N) - 1;
        } else if (P.stage_mode <= 1) {
            u64 used = 0;
            for (int i = 0; i < kNStagePrio && (P.stage_mode == 0 || i == 0); i++) {
                const int k = kStagePrio[i];
                const u64 b = im_round(s_sz[k]);
                if (used + b > P.stage_limit) continue;
                s_off[k] = used;
                used += b;
                mask |= 1u << k;
            }
        }
        V.staged = mask;
        for (int k = 0; k < IM_N; k++)
            set_slice(V, k, ((mask >> k) & 1) ? (const void *)(img + s_off[k])
                                              : global_slice(P, V.X, V.T, k));
    }
    __syncthreads();
    const u32 smask = V.staged;
    for (int k = 0; k < IM_N; k++)
        if ((smask >> k) & 1) block_copy(img + s_off[k], global_slice(P, V.X, V.T, k), s_sz[k]);
    __syncthreads();

    u32 t = TC.now0, status = TC.status0, left = TC.left0, now = TC.now0;
    const u64 lim64 = (u64)t + P.max_ticks;
    const u32 limit = lim64 > kTickLimit ? kTickLimit : (u32)lim64;
    u32 k = 0;
    if (status == EXP_RUNNING && left == 0) {
        status = EXP_DONE;
        now = TC.end_max1;
    }
    const u32 nI = V.X.n_items, nsw = V.X.nsw;
    // queue words in shared memory: a pass reads every free egress's
    // downstream queue words up front instead of after the plan
    const bool qstaged = ((smask >> IM_QPUSH) & (smask >> IM_QPOP) & 1u) != 0;
    const bool voq = V.X.voq != 0;      // switches keep virtual output queues
    // with DCQCN a warp forwards one switch a pass (marking reads the queue)
    const CcRec *ccr = (CC && V.X.cc) ? P.ccrec + (V.X.cc - 1) : nullptr;
    const bool onepass = voq || ccr != nullptr;
    // items are dealt to warps round-robin (item warp + j * nW), so switches
    // and rank groups spread over all warps
    const u32 cnt = warp < nI ? (nI - warp + nW - 1) / nW : 0;
    // Wake table: own[nI] (written by the item's warp only) and two poke
    // words per item.  Pokes made during step k go to word k & 1; the owner
    // folds them into own at the start of step k + 1, after the barrier, so
    // no poke is lost whatever order warps run in.  Pokes left by an earlier
    // run are folded before the first step.
    u32 *own = V.wake, *pk0 = V.wake + nI, *pk1 = V.wake + 2 * nI;
    for (u32 j = lane; j < cnt; j += 32) {
        const u32 it = warp + j * nW;
        u32 o = own[it], a = ld_vol32(&pk0[it]), b = ld_vol32(&pk1[it]);
        own[it] = min(o, min(a, b));
        pk0[it] = kUnset;
        pk1[it] = kUnset;
    }
    __syncthreads();
    Acc acc = {0, 0, 0, 0, 0, 0};
    bool now_end = false;              // the clock becomes 1 + the latest node end
    while (status == EXP_RUNNING) {
        if (t >= limit) { now = t; break; }
        u32 rep = kUnset, done = 0, fail = kUnset;
        u32 *poke = (k & 1) ? pk1 : pk0, *prev = (k & 1) ? pk0 : pk1;
        for (u32 base = 0; base < cnt; base += 32) {
            const u32 it = warp + (base + lane) * nW;
            u32 w = kUnset;
            if (base + lane < cnt) {
                w = own[it];
                const u32 q = ld_vol32(&prev[it]);
                if (q != kUnset) {
                    prev[it] = kUnset;
                    w = min(w, q);
                    own[it] = w;
                }
            }
            const bool due = w <= t;
            rep = min(rep, due ? kUnset : w);
            // due switches: the latency build steps them one a pass; the
            // occupancy build packs up to kPack switches and 64 ports a pass
            const bool dsw = due && it < nsw;
            if (kOnePerPass<VT>::value || onepass) {
                u32 Ms1 = __ballot_sync(kFull, dsw);
                while (Ms1) {
                    const u32 j = (u32)__ffs(Ms1) - 1;
                    Ms1 &= Ms1 - 1;
                    const u32 item = warp + (base + j) * nW;
                    const u32 old = __shfl_sync(kFull, w, j);
                    rep = min(rep, voq ? switch_voq<VT>(V, acc, item, t, old, poke, sm, &fail)
                                       : switch_tick<VT>(V, acc, item, t, old, poke, sm, &fail, qstaged,
                                                         ccr));
                }
            }
            uint2 sr = make_uint2(0, 0);
            if (dsw && !kOnePerPass<VT>::value && !onepass) sr = V.sw_rec[it];
            u32 Ms = (kOnePerPass<VT>::value || onepass) ? 0u : __ballot_sync(kFull, dsw);
            u32 n = 0, used = 0;
            while (Ms) {
                const u32 j = (u32)__ffs(Ms) - 1;
                Ms &= Ms - 1;
                const u32 np = __shfl_sync(kFull, sr.y, j), p0 = __shfl_sync(kFull, sr.x, j);
                const u32 old = __shfl_sync(kFull, w, j);
                if (n == kPack || used + np > kMaxPorts) {
                    rep = min(rep, switch_pack<VT>(V, acc, n, t, poke, sm, &fail, qstaged));
                    n = 0;
                    used = 0;
                }
                if (lane == 0) {
                    sm->sw[n] = warp + (base + j) * nW;
                    sm->base[n] = used;
                    sm->np[n] = np;
                    sm->p0[n] = p0;
                    sm->old[n] = old;
                }
                __syncwarp();
                n++;
                used += np;
            }
            if (n) rep = min(rep, switch_pack<VT>(V, acc, n, t, poke, sm, &fail, qstaged));
            // due rank groups, one a pass
            u32 Mr = __ballot_sync(kFull, due && it >= nsw);
            while (Mr) {
                const u32 j = (u32)__ffs(Mr) - 1;
                Mr &= Mr - 1;
                const u32 item = warp + (base + j) * nW;
                const u32 old = __shfl_sync(kFull, w, j);
                rep = min(rep, rank_tick<VT, CC>(P, V, TC, acc, item - nsw, t, old, poke, &done, &fail));
            }
        }
        rep = __reduce_min_sync(kFull, rep);
        if (lane == 0) {
            u32 ab = 0;
            if (warp == 0 && (k & 255) == 255) {
                if (ld_vol32(&P.glob->error)) ab = 1;
                else if (P.watchdog_ns && globaltimer() - t_start > P.watchdog_ns) {
                    atomicExch(&P.glob->error, 1u);
                    ab = 1;
                }
            }
            TC.rep[k & 1][warp] = make_uint4(rep, done, fail, ab);
        }
        __syncthreads();
        u32 nx = kUnset, dn = 0, fk = kUnset, ab = 0;
        for (u32 q = 0; q < nW; q++) {
            uint4 r = TC.rep[k & 1][q];
            nx = min(nx, r.x);
            dn += r.y;
            fk = min(fk, r.z);
            ab |= r.w;
        }
        left -= dn;
        k++;
        if (fk != kUnset) { status = fk & 7u; now_end = true; break; }
        if (left == 0) { status = EXP_DONE; now_end = true; break; }
        if (nx == kUnset) { status = EXP_DEADLOCK; now_end = true; break; }
        t = nx;
        if (ab) { now = t; break; }
    }
    for (int o = 16; o > 0; o >>= 1) {           // warp totals of the per-lane counters
        acc.inj += __shfl_xor_sync(kFull, acc.inj, o);
        acc.hops += __shfl_xor_sync(kFull, acc.hops, o);
        acc.del += __shfl_xor_sync(kFull, acc.del, o);
        acc.msg += __shfl_xor_sync(kFull, acc.msg, o);
        acc.dig += __shfl_xor_sync(kFull, acc.dig, o);
        acc.emax = max(acc.emax, __shfl_xor_sync(kFull, acc.emax, o));
    }
    if (lane == 0) {
        atomicAdd(&TC.pkts_injected, acc.inj);
        atomicAdd(&TC.pkt_hops, acc.hops);
        atomicAdd(&TC.pkts_delivered, acc.del);
        atomicAdd(&TC.msgs_delivered, acc.msg);
        atomicAdd(&TC.digest, acc.dig);
    }
    if (lane == 0 && acc.emax) atomicMax(&TC.end_max1, acc.emax);
    __syncthreads();
    if (now_end) now = TC.end_max1;
    for (int k2 = 0; k2 < IM_NDYN; k2++)            // dynamic arrays back to global memory
        if ((smask >> k2) & 1)
            block_copy(const_cast<void *>(global_slice(P, V.X, V.T, k2)), img + s_off[k2], s_sz[k2]);
    if (threadIdx.x == 0) {
        ExpCtl c;
        c.status = status;
        c.now = now;
        c.nodes_left = left;
        c.end_max1 = TC.end_max1;
        c.rec_count = TC.rec_count;
        c.pad0 = c.pad1 = c.pad2 = 0;
        c.pkts_injected = TC.pkts_injected;
        c.pkt_hops = TC.pkt_hops;
        c.pkts_delivered = TC.pkts_delivered;
        c.msgs_delivered = TC.msgs_delivered;
        c.digest = TC.digest;
        P.ctl[e] = c;
        atomicMax((unsigned long long *)&P.glob->steps, (unsigned long long)k);
    }
    __syncthreads();
}

// Persistent grid: each block takes the next experiment of the processing
// order until none is left (or the watchdog fired).  Builds (VAR): 1 lets a block
// use up to 255 registers a thread (lowest latency per tick, for
// experiments stepped from shared memory); MINB = 2 caps registers so two
// blocks share an SM (more experiments in flight, for experiments whose
// state stays in global memory and whose ticks wait on memory).  CC: with
// the DCQCN code (batches holding a DCQCN experiment).
template <int VAR, bool CC>
__global__ void __launch_bounds__(VAR == 4 ? 1024 : VAR == 3 ? 512 : 256, VAR == 2 ? 2 : 1)
k_megakernel(Params P)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    const u32 nW = blockDim.x >> 5, warp = threadIdx.x >> 5;
    SwSmem *sw = reinterpret_cast<SwSmem *>(dsm);
    unsigned char *img = dsm + nW * sizeof(SwSmem);
    const u64 t_start = globaltimer();
    for (;;) {
        if (threadIdx.x == 0) s_slot = ld_vol32(&P.glob->error) ? kUnset : atomicAdd(&P.glob->next, 1u);
        __syncthreads();
        const u32 slot = s_slot;
        __syncthreads();
        if (slot >= P.n_exps) break;
        run_experiment<typename ViewFor<VAR>::T, CC>(P, P.order[slot], img, sw + warp, t_start);
    }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_routes(const Params &p, u64 n_pairs_max, u32 level, cudaStream_t st)
{
    u64 blocks = (n_pairs_max + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks == 0) blocks = 1;
    k_routes<<<(unsigned)blocks, 256, 0, st>>>(p, level);
    return cudaGetLastError();
}

cudaError_t launch_up_lists(const Params &p, u32 n_sw_total, cudaStream_t st)
{
    u32 blocks = (n_sw_total + 255) / 256;
    k_up_lists<<<blocks ? (blocks > 1024 ? 1024 : blocks) : 1, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_init(const Params &p, u32 max_nodes, u32 max_queues, u32 max_ranks,
                        cudaStream_t st)
{
    u32 m = max_nodes > max_queues ? max_nodes : max_queues;
    m = m > max_ranks ? m : max_ranks;
    u32 bx = (m + 255) / 256;
    if (bx > 64) bx = 64;
    if (bx == 0) bx = 1;
    k_init_ctl<<<(p.n_exps + 255) / 256, 256, 0, st>>>(p);
    dim3 grid(bx, p.n_exps < 65535 ? p.n_exps : 65535);
    k_init<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_coll_times(const Params &p, u32 max_colls, cudaStream_t st)
{
    u32 bx = (max_colls + 255) / 256;
    bx = bx ? (bx > 256 ? 256 : bx) : 1;
    dim3 grid(bx, p.n_exps < 65535 ? p.n_exps : 65535);
    k_coll_times<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

u32 megakernel_smem(u32 warps, u32 image_bytes) { return warps * (u32)sizeof(SwSmem) + image_bytes; }

u32 megakernel_scratch_bytes() { return (u32)sizeof(SwSmem); }

template <int VAR>
static const void *megakernel_fn_of(bool cc)
{
    return cc ? (const void *)k_megakernel<VAR, true> : (const void *)k_megakernel<VAR, false>;
}

static const void *megakernel_fn(u32 variant, bool cc)
{
    return variant == 4 ? megakernel_fn_of<4>(cc)
         : variant == 3 ? megakernel_fn_of<3>(cc)
         : variant == 2 ? megakernel_fn_of<2>(cc) : megakernel_fn_of<1>(cc);
}

cudaError_t megakernel_prepare(u32 variant, bool cc, u32 warps, u32 smem_bytes,
                               int *blocks_per_sm, int *n_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const void *fn = megakernel_fn(variant, cc);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, (int)(warps * 32),
                                                         smem_bytes);
}

template <int VAR>
static void launch_variant(bool cc, const Params &p, u32 blocks, u32 warps, u32 smem_bytes,
                           cudaStream_t st)
{
    if (cc) k_megakernel<VAR, true><<<blocks, warps * 32, smem_bytes, st>>>(p);
    else k_megakernel<VAR, false><<<blocks, warps * 32, smem_bytes, st>>>(p);
}

cudaError_t launch_megakernel(u32 variant, bool cc, const Params &p, u32 blocks, u32 warps,
                              u32 smem_bytes, cudaStream_t st)
{
    if (variant == 4) launch_variant<4>(cc, p, blocks, warps, smem_bytes, st);
    else if (variant == 3) launch_variant<3>(cc, p, blocks, warps, smem_bytes, st);
    else if (variant == 2) launch_variant<2>(cc, p, blocks, warps, smem_bytes, st);
    else launch_variant<1>(cc, p, blocks, warps, smem_bytes, st);
    return cudaGetLastError();
}

}  // namespace mv
