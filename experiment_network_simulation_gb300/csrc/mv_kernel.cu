// mv_kernel.cu -- the persistent sm_103a megakernel of the SPME packet
// simulator, plus its set-up kernels.
//
// One launch advances every experiment of the batch (Multiverse section 4.3:
// all systems fused in one kernel, launched once per batch).  A grid-wide
// step processes one tick of every live experiment; each experiment keeps its
// own clock and skips ticks in which nothing can change.  Work items are
//   - one warp per (experiment, switch): plan + pull forwarding (section 4.2)
//     for up to 64 ports, staged in shared memory;
//   - one warp per (experiment, 32 ranks): DAG advance with the analytic
//     intra-server model (sections 3.2, 4.1), NIC injection, NIC receive and
//     acknowledgements.
// A single grid barrier separates steps.  Reads of state another entity may
// change in the same step see start-of-tick values: queue counters carry the
// tick of their last change (at most one push and one pop per queue and
// tick), start ticks are read as "joined before this tick", and completion
// counters are monotone with timestamped results.  That makes the parallel
// step equal to the serial phase order.
#include "mv_device.cuh"

namespace mv {

// ---------------------------------------------------------------- helpers
// splitmix64 finaliser (S. Vigna, splitmix64.c, public domain).
__device__ __forceinline__ u64 mix64(u64 z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}
__device__ __forceinline__ u64 cdiv(u64 a, u64 b) { return (a + b - 1) / b; }

__device__ __forceinline__ u64 ld_rlx64(const u64 *p)
{
    u64 v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_rlx64(u64 *p, u64 v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ u32 ld_rlx32(const u32 *p)
{
    u32 v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_rlx32(u32 *p, u32 v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ i32 ld_acq32(const i32 *p)
{
    i32 v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ u64 globaltimer()
{
    u64 t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(ExpCtl *c, u32 st, u32 k)
{
    atomicCAS(&c->status, (u32)EXP_RUNNING, st);
    atomicMin(&c->stop_step, k);
}

// Credit of queue qi for a sender at tick t: the queue holds `tail` pushes
// and `H` pops as of the start of the tick; the credit of a pop at tick x
// reaches the sender at x + D (D = delta + 1 of the link).  At most D - 1
// pops can still be on their way, so the pop log is only read when the
// queue is within D - 1 of full.
__device__ __forceinline__ bool credit_ok(const Params &P, u64 qi, u32 tail, u32 H, u32 D, u32 t,
                                          u32 cap)
{
    if (tail - H + D - 1 < cap) return true;
    u32 back = 0;
    const u32 *log = P.poplog + qi * kPopLog;
    while (back < H && back + 1 < D) {
        if (__ldcg(&log[(H - 1 - back) % kPopLog]) + D <= t) break;
        back++;
    }
    return tail - (H - back) < cap;
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

__global__ void k_up_lists(Params P, u32 n_sw_total)
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
    (void)n_sw_total;
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

// blockIdx.y = experiment; x covers that experiment's entities
__global__ void k_init(Params P)
{
    u32 e = blockIdx.y;
    const ExpRec X = P.exp[e];
    const WorkRec W = P.work[X.work];
    u32 i = blockIdx.x * blockDim.x + threadIdx.x;
    u32 stride = gridDim.x * blockDim.x;
    for (u32 u = i; u < X.nn; u += stride) {
        u64 g = X.nd_off + u;
        P.nd_pred[g] = P.node_npred[W.node_off + u];
        P.nd_cand[g] = 0;
        P.nd_start[g] = kUnset;
        P.nd_end[g] = kUnset;
        P.nd_pbase[g] = 0;
        P.nd_done[g] = 0;
        P.nd_out[g] = 0;
    }
    for (u32 q = i; q < X.nq; q += stride) {
        P.q_push[X.q_off + q] = (u64)kUnset << 32;
        P.q_pop[X.q_off + q] = (u64)kUnset << 32;
    }
    // work items: switches wake on their first packet, rank groups at tick 0
    for (u32 it = i; it < X.n_items; it += stride) P.wake[X.item_off + it] = it < X.nsw ? kUnset : 0;
    bool fits = memory_fits(P.mem + 10 * (u64)X.work, X.gpu_mem);
    // roots (no predecessor) are scheduled at tick 0, in node order
    for (u32 r = i; r < X.nr; r += stride) {
        RankCtl c = {};
        u32 first = P.rank_first[W.rank_off + r], cnt = P.rank_nnodes[W.rank_off + r];
        bool over = false;
        for (u32 u = first; u < first + cnt && fits; u++) {
            if (P.node_npred[W.node_off + u] != 0) continue;
            if (c.npend == kNPend) { over = true; break; }
            P.pend[(X.rk_off + r) * kNPend + c.npend++] = make_uint2(u, 0);
        }
        P.rk[X.rk_off + r] = c;
        if (over) atomicCAS(&P.ctl[e].status, (u32)EXP_RUNNING, (u32)EXP_OVERFLOW);
    }
}

__global__ void k_init_ctl(Params P)
{
    for (u32 e = blockIdx.x * blockDim.x + threadIdx.x; e < P.n_exps; e += gridDim.x * blockDim.x) {
        const ExpRec X = P.exp[e];
        ExpCtl c = {};
        c.status = memory_fits(P.mem + 10 * (u64)X.work, X.gpu_mem) ? EXP_RUNNING : EXP_OOM;
        c.now = 0;
        c.nodes_left = X.nn;
        c.stop_step = kUnset;
        P.ctl[e] = c;
    }
}

__global__ void k_run_reset(Params P, u32 max_ticks)
{
    for (u32 e = blockIdx.x * blockDim.x + threadIdx.x; e < P.n_exps; e += gridDim.x * blockDim.x) {
        ExpCtl *c = &P.ctl[e];
        c->stop_step = kUnset;
        u64 lim = (u64)c->now + max_ticks;
        c->limit = lim > kTickLimit ? kTickLimit : (u32)lim;
        for (int k = 0; k < 3; k++) {
            c->clk[k] = kUnset;
            c->nxt[k] = kUnset;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        Glob *g = P.glob;
        g->bar_count = 0;
        g->error = 0;
        g->run_cnt[0] = g->run_cnt[1] = g->run_cnt[2] = 0;
        g->steps = 0;
        g->err_step = g->err_block = kUnset;
    }
}

// ---------------------------------------------------------------- grid barrier
// Sense-counting barrier over all blocks of the cooperative launch.  Every
// wait is bounded by the run's timeout; past it the block records the error
// and leaves, and every block exits at its next barrier.
__device__ bool grid_barrier(const Params &P, u32 step)
{
    Glob *g = P.glob;
    __shared__ u32 ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        bool skip = (i32)blockIdx.x == P.fault_block && (i32)step == P.fault_step;
        u32 gen = ld_rlx32(&g->bar_gen);
        __threadfence();
        if (!skip) {
            u32 arrived = atomicAdd(&g->bar_count, 1);
            if (arrived == gridDim.x - 1) {
                g->bar_count = 0;
                __threadfence();
                atomicAdd(&g->bar_gen, 1);
            }
        }
        if (ld_rlx32(&g->bar_gen) == gen) {
            u64 t0 = globaltimer();
            u32 it = 0;
            while (ld_rlx32(&g->bar_gen) == gen) {
                if (ld_rlx32(&g->error)) { ok = 0; break; }
                if ((++it & 255) == 0 && globaltimer() - t0 > P.barrier_timeout_ns) {
                    if (atomicCAS(&g->error, 0u, 1u) == 0) {
                        g->err_step = step;
                        g->err_block = blockIdx.x;
                    }
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        if (ld_rlx32(&g->error)) ok = 0;
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

// ---------------------------------------------------------------- clocks
// Tick that experiment e processes at step k, or kUnset if it does not run.
// Every lane that touches e computes it the same way, from the slots of step
// k-1 only: the clock and the minimum over every pending wake tick reported
// during step k-1 (three rotating slots: step k-1's are stable while step k
// runs, and step k+1's are cleared during step k).
__device__ __forceinline__ u32 exp_tick(const Params &P, u32 e, u32 k)
{
    ExpCtl *c = &P.ctl[e];
    u32 stop = ld_rlx32(&c->stop_step), lim = ld_rlx32(&c->limit);
    if (stop < k) return kUnset;                  // finished or failed earlier
    u32 t;
    if (k == 0) {
        u32 st = ld_rlx32(&c->status), left = ld_rlx32(&c->nodes_left);
        t = ld_rlx32(&c->now);
        if (st != EXP_RUNNING || left == 0) return kUnset;
    } else {
        u32 p = (k - 1) % 3;
        u32 tp = ld_rlx32(&c->clk[p]);
        t = ld_rlx32(&c->nxt[p]);
        if (tp == kUnset || t == kUnset) return kUnset;
    }
    return t >= lim ? kUnset : t;
}

// Control of one experiment at step k (run by the lane holding its first
// work item): publish its tick, clear the slot of step k+1, count it as
// running, and settle its final state when it stops.
__device__ void exp_control(const Params &P, u32 e, u32 k, u32 t)
{
    ExpCtl *c = &P.ctl[e];
    st_rlx32(&c->clk[k % 3], t);
    st_rlx32(&c->nxt[(k + 1) % 3], kUnset);
    if (t != kUnset) {
        atomicAdd(&P.glob->run_cnt[k % 3], 1);
        return;
    }
    // a stopped experiment's clock is one past its latest node end (0: none)
    if (k == 0) {
        if (ld_rlx32(&c->status) == EXP_RUNNING && ld_rlx32(&c->nodes_left) == 0) {
            st_rlx32(&c->status, EXP_DONE);
            st_rlx32(&c->now, ld_rlx32(&c->end_max1));
        }
        return;                                   // else stopped before: now unchanged
    }
    u32 p = (k - 1) % 3, tp = ld_rlx32(&c->clk[p]);
    if (tp == kUnset) return;                     // settled at an earlier step
    u32 nx = ld_rlx32(&c->nxt[p]);
    if (ld_rlx32(&c->status) != EXP_RUNNING) {    // failed during the last tick
        st_rlx32(&c->now, ld_rlx32(&c->end_max1));
    } else if (ld_rlx32(&c->nodes_left) == 0) {
        st_rlx32(&c->status, EXP_DONE);
        st_rlx32(&c->now, ld_rlx32(&c->end_max1));
    } else if (nx == kUnset) {                    // nothing pending anywhere
        st_rlx32(&c->status, EXP_DEADLOCK);
        st_rlx32(&c->now, ld_rlx32(&c->end_max1));
    } else {                                      // stopped by the tick budget
        st_rlx32(&c->now, nx);
    }
}

// Work items and their wake ticks.  An item is processed at tick t when its
// wake <= t.  Whoever creates work for another item lowers that item's wake
// (a push, a collective join, a message delivery) and the experiment's next
// tick; a processed item sets its own next wake from its own state.
__device__ __forceinline__ u32 sw_item(const ExpRec &X, u32 s) { return X.item_off + s; }
__device__ __forceinline__ u32 rank_item(const ExpRec &X, u32 r) { return X.item_off + X.nsw + r / 32; }
__device__ __forceinline__ void poke(const Params &P, u32 item, u32 e, u32 k, u32 at)
{
    atomicMin(&P.wake[item], at);
    atomicMin(&P.ctl[e].nxt[k % 3], at);
}

// ---------------------------------------------------------------- switches
struct SwSmem {
    uint4 pkt[kMaxPorts];
    unsigned long long mask[kMaxPorts];
    u32 head[kMaxPorts];
    u32 pad[2];
};

__device__ __forceinline__ u32 route_port(const Params &P, const TopoRec &T, const ExpRec &X,
                                          u32 gs, u32 s, uint4 pk)
{
    u8 r = P.route[T.route_off + (u64)s * T.nh + pk_dst(pk)];
    if (r != 0xFF) return r;
    u32 nup = P.up_n[gs];
    if (nup == 0) return 0xFFu;
    u64 h = mix64((u64)pk_key(pk) ^ ((u64)s << 40) ^ X.ecmp_seed);
    return P.up_list[T.port_off + P.sw_pstart[gs] + (u32)(h % nup)];
}

// Forwarding at one switch for one tick (Multiverse section 4.2): each lane
// plans its ingress ports (the egress their ready head packet needs), then
// each lane pulls for its egress ports: free link, credit downstream, first
// planned ingress at or after the round-robin pointer.
__device__ void switch_tick(const Params &P, const ExpRec &X, u32 e, u32 s, u32 t, u32 k,
                            SwSmem *sm)
{
    const TopoRec T = P.topo[X.topo];
    const u32 lane = threadIdx.x & 31;
    const u32 gs = T.sw_off + s;
    const u32 np = P.sw_nports[gs], p0 = P.sw_pstart[gs];
    const u32 it = sw_item(X, s);
    u32 old = 0;
    if (lane == 0) old = atomicExch(&P.wake[it], kUnset);   // consume pending wakes
    old = __shfl_sync(0xffffffffu, old, 0);
    u32 nxt = kUnset;                   // own next wake
    u32 pk_min = kUnset;                // earliest tick poked into a downstream item
    bool ready_any = false;
    bool bad = false;
    sm->mask[lane] = 0;
    sm->mask[lane + 32] = 0;
    __syncwarp();
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        u32 p = lane + 32 * j;
        if (p >= np) continue;
        u64 qi = X.q_off + p0 + p;
        u64 pw = ld_rlx64(&P.q_push[qi]);
        u32 tail = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
        u32 head = (u32)__ldcg(&P.q_pop[qi]);
        sm->head[p] = head;
        if (head == tail) continue;
        uint4 pk = __ldcg(&P.slots[X.slot_off + (u64)(p0 + p) * X.cap + head % X.cap]);
        if (pk.x > t) { nxt = min(nxt, pk.x); continue; }
        ready_any = true;
        u32 tg = route_port(P, T, X, gs, s, pk);
        if (tg >= np) { bad = true; continue; }
        sm->pkt[p] = pk;
        atomicOr(&sm->mask[tg], 1ull << p);
    }
    __syncwarp();
    unsigned long long popped = 0;
    u32 hops = 0;
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        u32 eg = lane + 32 * j;
        if (eg >= np) continue;
        unsigned long long M = sm->mask[eg];
        if (!M) continue;
        u32 qe = p0 + eg;
        uint2 st = __ldcg(&P.eg[X.eg_off + qe]);
        if (st.x > t) continue;             // busy: its heads wake the switch at t+1
        i32 pe = P.port_peer[T.port_off + qe];
        u32 dq = pe >= 0 ? (u32)pe : T.nq + (u32)(-pe - 1);
        u64 dqi = X.q_off + dq;
        u64 dpop = ld_rlx64(&P.q_pop[dqi]);
        u32 dhead = (u32)dpop - ((u32)(dpop >> 32) == t ? 1u : 0u);
        u32 dtail = (u32)__ldcg(&P.q_push[dqi]);
        u32 dl_e = P.port_delta[T.port_off + qe];
        if (!credit_ok(P, dqi, dtail, dhead, dl_e + 1, t, X.cap)) continue;
        unsigned long long hi = st.y < 64 ? (M & (~0ull << st.y)) : 0ull;
        u32 i = (u32)__ffsll((long long)(hi ? hi : M)) - 1;
        uint4 pk = sm->pkt[i];
        u32 sg = P.port_sigma[T.port_off + qe], dl = P.port_delta[T.port_off + qe];
        pk.x = t + sg + dl;
        pk.y += (dl + 1) << 16;
        __stcg(&P.slots[X.slot_off + (u64)dq * X.cap + dtail % X.cap], pk);
        st_rlx64(&P.q_push[dqi], ((u64)t << 32) | (u32)(dtail + 1));
        __stcg(&P.eg[X.eg_off + qe], make_uint2(t + sg, (i + 1) % np));
        // the queue's owner: the peer switch, or the rank group of the host
        if (pe >= 0) atomicMin(&P.wake[sw_item(X, P.port_sw[T.port_off + pe])], pk.x);
        else if ((u32)(-pe - 1) < X.nr) atomicMin(&P.wake[rank_item(X, (u32)(-pe - 1))], pk.x);
        pk_min = min(pk_min, pk.x);
        popped |= 1ull << i;
        hops++;
    }
    u32 lo = __reduce_or_sync(0xffffffffu, (u32)popped);
    u32 hi32 = __reduce_or_sync(0xffffffffu, (u32)(popped >> 32));
    unsigned long long all = ((unsigned long long)hi32 << 32) | lo;
#pragma unroll
    for (u32 j = 0; j < 2; j++) {
        u32 p = lane + 32 * j;
        if (p < np && ((all >> p) & 1ull)) {
            u64 qi = X.q_off + p0 + p;
            __stcg(&P.poplog[qi * kPopLog + sm->head[p] % kPopLog], t);
            st_rlx64(&P.q_pop[qi], ((u64)t << 32) | (u32)(sm->head[p] + 1));
        }
    }
    hops = __reduce_add_sync(0xffffffffu, hops);
    nxt = __reduce_min_sync(0xffffffffu, nxt);
    pk_min = __reduce_min_sync(0xffffffffu, pk_min);
    bool anybad = __any_sync(0xffffffffu, bad);
    if (__any_sync(0xffffffffu, ready_any)) nxt = t + 1;   // heads left or blocked
    if (lane == 0) {
        ExpCtl *c = &P.ctl[e];
        u32 w = min(nxt, old > t ? old : kUnset);
        if (w != kUnset) atomicMin(&P.wake[it], w);
        u32 m = min(w, pk_min);
        if (m != kUnset) atomicMin(&c->nxt[k % 3], m);
        if (all) atomicAdd((unsigned long long *)&c->pkt_hops, (unsigned long long)hops);
        if (anybad) set_status(c, EXP_ERROR, k);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- ranks
// Rank state goes through L2 (.cg): the item of a rank always lands on the
// same warp, but state written by set-up kernels must not come from L1.
__device__ __forceinline__ RankCtl load_ctl(const RankCtl *p)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    uint4 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
    RankCtl r;
    r.busy = a.x; r.rr = a.y; r.npend = a.z; r.nact = a.w;
    r.lane_mask = ((u64)b.y << 32) | b.x;
    r.port_mask[0] = ((u64)b.w << 32) | b.z;
    r.port_mask[1] = ((u64)c.y << 32) | c.x;
    r.pad = 0;
    return r;
}
__device__ __forceinline__ void store_ctl(RankCtl *p, const RankCtl &r)
{
    uint4 *q = reinterpret_cast<uint4 *>(p);
    __stcg(q, make_uint4(r.busy, r.rr, r.npend, r.nact));
    __stcg(q + 1, make_uint4((u32)r.lane_mask, (u32)(r.lane_mask >> 32), (u32)r.port_mask[0],
                             (u32)(r.port_mask[0] >> 32)));
    __stcg(q + 2, make_uint4((u32)r.port_mask[1], (u32)(r.port_mask[1] >> 32), 0, 0));
}
__device__ __forceinline__ Lane load_lane(const Lane *p)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    Lane L;
    uint4 *d = reinterpret_cast<uint4 *>(&L);
    d[0] = __ldcg(q); d[1] = __ldcg(q + 1); d[2] = __ldcg(q + 2); d[3] = __ldcg(q + 3);
    return L;
}
__device__ __forceinline__ void store_lane(Lane *p, const Lane &L)
{
    uint4 *q = reinterpret_cast<uint4 *>(p);
    const uint4 *s = reinterpret_cast<const uint4 *>(&L);
    __stcg(q, s[0]); __stcg(q + 1, s[1]); __stcg(q + 2, s[2]); __stcg(q + 3, s[3]);
}

// Per-rank view used while processing one tick.
struct RankView {
    const Params *P;
    const ExpRec *X;
    const TopoRec *T;
    const WorkRec *W;
    ExpCtl *c;
    u32 r, t, e, k;
    u64 rk;             // X.rk_off + r
    RankCtl C;
    bool changed, fail_over, fail_err;
    u32 nxt;            // this rank's own next wake
    u32 pk_min;         // earliest wake poked into other items
    u32 n_inj, n_del, n_msg, n_done, end_max1;
    u64 dig;
};

__device__ __forceinline__ u32 coll_of(const RankView &v, u32 u) { return v.P->node_arg[v.W->node_off + u]; }
__device__ __forceinline__ u32 nmemb(const RankView &v, u32 c) { return v.P->coll_nmembers[v.W->coll_off + c]; }
__device__ __forceinline__ u32 ckind(const RankView &v, u32 c) { return v.P->coll_kind[v.W->coll_off + c]; }
__device__ __forceinline__ u64 cbytes(const RankView &v, u32 c) { return v.P->coll_bytes[v.W->coll_off + c]; }
__device__ __forceinline__ u32 mabs(const RankView &v, u32 c, u32 i)
{
    return v.W->memb_off + v.P->coll_mstart[v.W->coll_off + c] + i;
}
__device__ __forceinline__ u32 mrank(const RankView &v, u32 c, u32 i) { return v.P->member_rank[mabs(v, c, i)]; }
__device__ __forceinline__ u32 mnode(const RankView &v, u32 c, u32 i) { return v.P->member_node[mabs(v, c, i)]; }
__device__ __forceinline__ bool tree_of(const RankView &v, u32 c)
{
    return ckind(v, c) == COLL_AR && v.X->algo == ALGO_TREE;
}
__device__ __forceinline__ u32 nchan(const RankView &v, u32 c)
{
    u32 k = ckind(v, c);
    return (k == COLL_RELAY || k == COLL_P2P) ? 1u : v.X->nc;
}
__device__ __forceinline__ u32 nports_of(const RankView &v, u32 c)
{
    u32 k = ckind(v, c);
    if (k == COLL_RELAY || k == COLL_P2P || k == COLL_A2A) return 1;
    return nchan(v, c) * (tree_of(v, c) ? 3u : 1u);
}
// channel c's share of S bytes (AutoCCL section 2.3: NC partitions)
__device__ __forceinline__ u64 part_bytes(u64 S, u32 nc, u32 c) { return S / nc + (c < S % nc ? 1 : 0); }
__device__ __forceinline__ u64 nchunks(u64 b, u64 C) { return b == 0 ? 1 : cdiv(b, C); }
__device__ __forceinline__ u32 ring_steps(const RankView &v, u32 c)
{
    u32 N = nmemb(v, c);
    if (N < 2) return 0;
    return ckind(v, c) == COLL_AR ? 2 * (N - 1) : N - 1;
}
__device__ __forceinline__ u64 ring_loops(const RankView &v, u32 c, u64 Pc)
{
    return Pc == 0 ? 1 : cdiv(Pc, (u64)nmemb(v, c) * v.X->chunk);
}
__device__ u64 a2a_row_chunks(const RankView &v, u32 c, u32 i)
{
    u32 m = mabs(v, c, i);
    u32 b = v.W->a2a_off + v.P->memb_row[m], n = v.P->member_a2a_n[m];
    u64 tot = 0;
    for (u32 j = 0; j < n; j++) tot += nchunks(v.P->a2a_bytes[b + j], v.X->chunk);
    return tot;
}

__device__ u32 lane_count(const RankView &v, u32 c, u32 i, u32 ch, u32 kind)
{
    u32 N = nmemb(v, c);
    u64 S = cbytes(v, c);
    switch (ckind(v, c)) {
    case COLL_AR: case COLL_RS: case COLL_AG:
        if (tree_of(v, c)) {
            u64 n = nchunks(part_bytes(S, v.X->nc, ch), v.X->chunk);
            if (kind == 0) return i > 0 ? (u32)n : 0;
            return 2 * i + kind < N ? (u32)n : 0;
        }
        return (u32)(ring_loops(v, c, part_bytes(S, v.X->nc, ch)) * ring_steps(v, c));
    case COLL_RELAY:
        return i + 1 < N ? v.P->coll_parts[v.W->coll_off + c] : 0;
    case COLL_P2P:
        return i == 0 ? (u32)nchunks(S, v.X->chunk) : 0;
    case COLL_A2A: {
        u64 tot = a2a_row_chunks(v, c, i);
        return tot > ch ? (u32)cdiv(tot - ch, v.X->nc) : 0;
    }
    }
    return 0;
}

__device__ u32 port_count_expect(const RankView &v, u32 c, u32 i, u32 p)
{
    u32 N = nmemb(v, c);
    u64 S = cbytes(v, c);
    switch (ckind(v, c)) {
    case COLL_AR: case COLL_RS: case COLL_AG:
        if (tree_of(v, c)) {
            u32 ch = p / 3, q = p % 3;
            u64 n = nchunks(part_bytes(S, v.X->nc, ch), v.X->chunk);
            if (q == 0) return i > 0 ? (u32)n : 0;
            return 2 * i + q < N ? (u32)n : 0;
        }
        return (u32)(ring_loops(v, c, part_bytes(S, v.X->nc, p)) * ring_steps(v, c));
    case COLL_RELAY:
        return i > 0 ? v.P->coll_parts[v.W->coll_off + c] : 0;
    case COLL_P2P:
        return i == 1 ? (u32)nchunks(S, v.X->chunk) : 0;
    case COLL_A2A: {
        u32 m = mabs(v, c, i);
        u32 b = v.W->a2a_in_off + v.P->memb_col[m], n = v.P->member_a2a_in_n[m];
        u64 tot = 0;
        for (u32 j = 0; j < n; j++) tot += nchunks(v.P->a2a_in_bytes[b + j], v.X->chunk);
        return (u32)tot;
    }
    }
    return 0;
}

// Message L.m of a lane: bytes, destination member and port, and the own
// receive counts it waits for.  Returns its packet count.
__device__ u32 lane_setup(const RankView &v, Lane &L)
{
    u32 c = coll_of(v, L.node), N = nmemb(v, c), i = L.member, m = L.m, ch = L.chan;
    u64 S = cbytes(v, c), C = v.X->chunk, bytes = 0;
    L.dep_mask = 0;
    L.dep_need = 0;
    L.dep_base = 0;
    switch (ckind(v, c)) {
    case COLL_AR: case COLL_RS: case COLL_AG: {
        u64 Pc = part_bytes(S, v.X->nc, ch);
        if (tree_of(v, c)) {
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
            u32 steps = ring_steps(v, c);
            u64 l = m / steps, kk = m % steps, stride = (u64)N * C;
            u64 B = min(stride, Pc - l * stride);
            u64 bs = cdiv(B, N);
            u64 blk = ((u64)i + N - (kk % N)) % N;
            bytes = B > blk * bs ? min(bs, B - blk * bs) : 0;
            L.dst_member = (i + 1) % N;
            L.dst_port = ch;
            L.dep_base = ch;
            if (kk >= 1) { L.dep_mask = 1u; L.dep_need = (u32)(l * steps + kk); }
        }
        break;
    }
    case COLL_RELAY: {                                // pipelined broadcast hop
        u32 K = v.P->coll_parts[v.W->coll_off + c];
        bytes = S / K + (m < S % K ? 1 : 0);
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
        u32 mm = mabs(v, c, i);
        u32 r0 = v.W->a2a_off + v.P->memb_row[mm];
        u64 g = (u64)ch + (u64)m * v.X->nc;
        while (g >= L.a2a_start + nchunks(v.P->a2a_bytes[r0 + L.a2a_e], C)) {
            L.a2a_start += (u32)nchunks(v.P->a2a_bytes[r0 + L.a2a_e], C);
            L.a2a_e++;
        }
        u64 j = g - L.a2a_start, b = v.P->a2a_bytes[r0 + L.a2a_e];
        bytes = b > j * C ? min(C, b - j * C) : 0;
        L.dst_member = v.P->a2a_dst[r0 + L.a2a_e];
        L.dst_port = 0;
        break;
    }
    }
    u32 drank = mrank(v, c, L.dst_member);
    L.key = (u32)(mix64((u64)L.node | ((u64)(ch * 4 + L.kind) << 32) | ((u64)drank << 44)) &
                  0xFFFFFFu);
    return (u32)(bytes == 0 ? 1 : cdiv(bytes, v.X->pkt));
}

__device__ u32 compute_ticks(const RankView &v, u32 u)
{
    const Params &P = *v.P;
    u64 lo = P.node_dur_lo[v.W->node_off + u], hi = P.node_dur_hi[v.W->node_off + u], ns = lo;
    if (hi > lo)
        ns = lo + mix64(mix64((u64)P.node_dur_key[v.W->node_off + u]) ^ v.X->dur_seed) % (hi - lo + 1);
    return (u32)cdiv(ns * 1000, v.X->tick_ps);
}

// alpha + bytes/beta (Multiverse section 4.1), beta as ticks per byte
__device__ u32 intra_ticks(const RankView &v, u32 c)
{
    const Params &P = *v.P;
    u32 cc = v.W->coll_off + c;
    u64 g = nmemb(v, c), S = cbytes(v, c), be;
    switch (ckind(v, c)) {
    case COLL_AR: be = cdiv(2 * (g - 1) * S, g); break;
    case COLL_RS: case COLL_AG: be = cdiv((g - 1) * S, g); break;
    default: be = S;
    }
    return P.coll_alpha[cc] + (u32)cdiv(be * P.coll_beta_num[cc], P.coll_beta_den[cc]);
}

__device__ __forceinline__ void rank_poke(RankView &v, u32 item, u32 at)
{
    atomicMin(&v.P->wake[item], at);
    v.pk_min = min(v.pk_min, at);
}

// A member joined collective c at this tick: members waiting on its start
// look again when the join reaches them (intra-server barrier: next tick;
// network rendezvous: 1 + min(delta) ticks later).
__device__ void poke_members(RankView &v, u32 c, u32 at)
{
    u32 N = nmemb(v, c), last = kUnset;
    for (u32 m = 0; m < N; m++) {
        u32 g = rank_item(*v.X, mrank(v, c, m));
        if (g != last) rank_poke(v, g, at);
        last = g;
    }
}

__device__ void pend_add(RankView &v, u32 u, u32 st)
{
    if (v.C.npend >= kNPend) { v.fail_over = true; return; }
    v.P->pend[v.rk * kNPend + v.C.npend++] = make_uint2(u, st);
}

__device__ void complete_node(RankView &v, u32 u, u32 c)
{
    const Params &P = *v.P;
    u64 g = v.X->nd_off + u;
    __stcg(&P.nd_end[g], c);
    v.n_done++;
    v.end_max1 = max(v.end_max1, c + 1);
    v.changed = true;
    if (c >= kTickLimit) { v.fail_over = true; return; }
    u32 s0 = P.succ_start[v.W->node_off + u], ns = P.node_nsucc[v.W->node_off + u];
    for (u32 j = 0; j < ns; j++) {
        u32 w = P.succ[v.W->edge_off + s0 + j];
        u64 gw = v.X->nd_off + w;
        u32 cd = max(__ldcg(&P.nd_cand[gw]), c + 1);
        __stcg(&P.nd_cand[gw], cd);
        u32 left = __ldcg(&P.nd_pred[gw]) - 1;
        __stcg(&P.nd_pred[gw], left);
        if (left == 0) pend_add(v, w, cd);
    }
}

__device__ void free_ports(RankView &v, u32 u)
{
    u32 np = nports_of(v, coll_of(v, u)), b = __ldcg(&v.P->nd_pbase[v.X->nd_off + u]);
    for (u32 p = b; p < b + np; p++) v.C.port_mask[p >> 6] &= ~(1ull << (p & 63));
}

// A rank joins a network collective: receive counters, then send lanes.
__device__ bool net_join(RankView &v, u32 u)
{
    const Params &P = *v.P;
    u32 c = coll_of(v, u), i = P.node_member[v.W->node_off + u];
    u32 np = nports_of(v, c);
    i32 base = -1;
    for (u32 b = 0; b + np <= kNPort && base < 0; b++) {
        u32 k = 0;
        while (k < np && !((v.C.port_mask[(b + k) >> 6] >> ((b + k) & 63)) & 1ull)) k++;
        if (k == np) base = (i32)b;
    }
    if (base < 0) { v.fail_over = true; return false; }
    i32 out = 0;
    for (u32 p = 0; p < np; p++) {
        u32 s = (u32)base + p;
        v.C.port_mask[s >> 6] |= 1ull << (s & 63);
        P.ports[v.rk * kNPort + s] = make_uint2(0, u);
        out += (i32)port_count_expect(v, c, i, p);
    }
    u32 nch = nchan(v, c), lpc = tree_of(v, c) ? 3u : 1u;
    for (u32 ch = 0; ch < nch; ch++) {
        for (u32 kd = 0; kd < lpc; kd++) {
            u32 nm = lane_count(v, c, i, ch, kd);
            if (nm == 0) continue;
            u64 freem = ~v.C.lane_mask;
            if (!freem) { v.fail_over = true; return false; }
            u32 slot = (u32)__ffsll((long long)freem) - 1;
            Lane L = {};
            L.node = u; L.member = i; L.chan = ch; L.kind = kd;
            L.m = 0; L.nmsg = nm;
            L.pkts_left = lane_setup(v, L);
            store_lane(&P.lanes[v.rk * kNLane + slot], L);
            v.C.lane_mask |= 1ull << slot;
            out += (i32)nm;
        }
    }
    u64 g = v.X->nd_off + u;
    __stcg(&P.nd_pbase[g], (u32)base);
    __stcg(&P.nd_done[g], v.t);
    __stcg(&P.nd_out[g], out);
    return true;
}

__device__ void act_add(RankView &v, u32 u)
{
    if (v.C.nact >= kNAct) { v.fail_over = true; return; }
    u32 *a = v.P->act + v.rk * kNAct;
    u32 j = v.C.nact;                       // keep ascending node order
    while (j > 0 && __ldcg(&a[j - 1]) > u) { __stcg(&a[j], __ldcg(&a[j - 1])); j--; }
    __stcg(&a[j], u);
    v.C.nact++;
}

// Schedule + AnalyticalSys: finish running memberships, then start the nodes
// scheduled for this tick (both in node order).
__device__ void dag_step(RankView &v)
{
    const Params &P = *v.P;
    const u32 t = v.t;
    u32 *a = P.act + v.rk * kNAct;
    u32 w = 0;
    for (u32 j = 0; j < v.C.nact; j++) {
        u32 u = __ldcg(&a[j]), c = coll_of(v, u);
        bool fin = false;
        if (P.node_kind[v.W->node_off + u] == NODE_INTRA) {
            u32 N = nmemb(v, c), b = 0;
            bool ok = true;
            for (u32 m = 0; m < N && ok; m++) {
                u32 st = ld_rlx32(&P.nd_start[v.X->nd_off + mnode(v, c, m)]);
                if (st == kUnset || st >= t) ok = false;
                else b = max(b, st);
            }
            if (ok) { complete_node(v, u, b + intra_ticks(v, c)); fin = true; }
        } else {
            u64 g = v.X->nd_off + u;
            if (ld_acq32(&P.nd_out[g]) == 0) {
                u32 done = ld_rlx32(&P.nd_done[g]);
                free_ports(v, u);
                complete_node(v, u, done);
                fin = true;
            }
        }
        if (!fin) __stcg(&a[w++], u);
    }
    v.C.nact = w;
    // start scheduled nodes: take those due now out of the pending list
    uint2 *pd = P.pend + v.rk * kNPend;
    u32 due[kNPend];
    u32 nd = 0, keep = 0;
    for (u32 j = 0; j < v.C.npend; j++) {
        uint2 x = __ldcg(&pd[j]);
        if (x.y < t) { v.fail_err = true; continue; }
        if (x.y == t) due[nd++] = x.x;
        else { __stcg(&pd[keep++], x); v.nxt = min(v.nxt, x.y); }
    }
    v.C.npend = keep;
    for (u32 j = 1; j < nd; j++) {           // insertion sort, node order
        u32 x = due[j], q = j;
        while (q > 0 && due[q - 1] > x) { due[q] = due[q - 1]; q--; }
        due[q] = x;
    }
    for (u32 j = 0; j < nd; j++) {
        u32 u = due[j];
        u64 g = v.X->nd_off + u;
        v.changed = true;
        u32 kind = P.node_kind[v.W->node_off + u];
        if (kind == NODE_COMPUTE) {
            __stcg(&P.nd_start[g], t);
            complete_node(v, u, t + compute_ticks(v, u));
        } else if (kind == NODE_INTRA) {
            st_rlx32(&P.nd_start[g], t);
            act_add(v, u);
            poke_members(v, coll_of(v, u), t + 1);
        } else {
            if (!net_join(v, u)) return;
            st_rlx32(&P.nd_start[g], t);
            poke_members(v, coll_of(v, u), t + v.T->rdv);
            if (__ldcg(&P.nd_out[g]) == 0) {
                free_ports(v, u);
                complete_node(v, u, t);
            } else {
                act_add(v, u);
            }
        }
        if (v.fail_over || v.fail_err) return;
    }
    // nodes scheduled by completions above may start later; note the earliest
    for (u32 j = 0; j < v.C.npend; j++) v.nxt = min(v.nxt, __ldcg(&pd[j]).y);
}

// SendSys + NICSndSys: one packet per uplink serialisation time, round-robin
// over the send lanes from the pointer; a lane is eligible once its receive
// dependencies are met and its destination joined before this tick.
__device__ void inject(RankView &v)
{
    const Params &P = *v.P;
    const u32 t = v.t;
    if (!v.C.lane_mask) return;
    if (v.C.busy > t) { v.nxt = min(v.nxt, v.C.busy); return; }
    const TopoRec &T = *v.T;
    u32 qp = P.host_port[T.host_off + v.r];
    u64 qi = v.X->q_off + qp;
    u64 pw = ld_rlx64(&P.q_pop[qi]);
    u32 head = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
    u32 tail = (u32)__ldcg(&P.q_push[qi]);
    if (!credit_ok(P, qi, tail, head, P.host_delta[T.host_off + v.r] + 1, t, v.X->cap)) {
        v.nxt = min(v.nxt, t + 1);
        return;
    }
    u64 M = v.C.lane_mask;
    u64 hi = v.C.rr < 64 ? (M & (~0ull << v.C.rr)) : 0ull;
    u64 lo = M & ~hi;
    Lane *lanes = P.lanes + v.rk * kNLane;
    for (int pass = 0; pass < 2; pass++) {
        u64 m = pass == 0 ? hi : lo;
        while (m) {
            u32 l = (u32)__ffsll((long long)m) - 1;
            m &= m - 1;
            Lane L = load_lane(&lanes[l]);
            u32 pb = __ldcg(&P.nd_pbase[v.X->nd_off + L.node]);
            bool ok = true;
            for (u32 b = 0; b < 3 && ok; b++)
                if ((L.dep_mask >> b) & 1u)
                    if (__ldcg(&P.ports[v.rk * kNPort + pb + L.dep_base + b]).x < L.dep_need) ok = false;
            if (!ok) continue;
            u32 c = coll_of(v, L.node);
            u64 dg = v.X->nd_off + mnode(v, c, L.dst_member);
            u32 dst_start = ld_rlx32(&P.nd_start[dg]);
            // the destination's join reaches this rank 1 + min(delta) ticks
            // later; when that time is known, it is this rank's own wake (a
            // poke alone could be shadowed by an earlier pending wake)
            if (dst_start == kUnset) continue;
            if (dst_start + T.rdv > t) { v.nxt = min(v.nxt, dst_start + T.rdv); continue; }
            u32 dpb = ld_rlx32(&P.nd_pbase[dg]);
            u32 hs = P.host_sigma[T.host_off + v.r], hd = P.host_delta[T.host_off + v.r];
            uint4 pk;
            pk.x = t + hs + hd;
            pk.y = mrank(v, c, L.dst_member) | ((hd + 1) << 16);
            pk.z = L.node;
            pk.w = L.key | ((L.pkts_left == 1 ? 1u : 0u) << 24) | ((dpb + L.dst_port) << 25);
            __stcg(&P.slots[v.X->slot_off + (u64)qp * v.X->cap + tail % v.X->cap], pk);
            st_rlx64(&P.q_push[qi], ((u64)t << 32) | (u32)(tail + 1));
            v.C.busy = t + hs;
            v.C.rr = (l + 1) % kNLane;
            v.n_inj++;
            v.changed = true;
            rank_poke(v, sw_item(*v.X, P.port_sw[T.port_off + qp]), pk.x);
            if (--L.pkts_left == 0) {
                if (++L.m == L.nmsg) v.C.lane_mask &= ~(1ull << l);
                else L.pkts_left = lane_setup(v, L);
            }
            store_lane(&lanes[l], L);
            if (v.C.lane_mask) v.nxt = min(v.nxt, v.C.busy > t + 1 ? v.C.busy : t + 1);
            return;
        }
    }
}

// NICRcvSys + ACKSys: take the ready head of the downlink queue; the last
// packet of a message completes it at this rank and acknowledges it to the
// sender, sum over hops of (delta + 1) ticks later.
__device__ void receive(RankView &v)
{
    const Params &P = *v.P;
    const u32 t = v.t;
    u32 ql = v.T->nq + v.r;
    u64 qi = v.X->q_off + ql;
    u64 pw = ld_rlx64(&P.q_push[qi]);
    u32 tail = (u32)pw - ((u32)(pw >> 32) == t ? 1u : 0u);
    u32 head = (u32)__ldcg(&P.q_pop[qi]);
    if (head == tail) return;
    uint4 pk = __ldcg(&P.slots[v.X->slot_off + (u64)ql * v.X->cap + head % v.X->cap]);
    if (pk.x > t) { v.nxt = min(v.nxt, pk.x); return; }
    __stcg(&P.poplog[qi * kPopLog + head % kPopLog], t);
    st_rlx64(&P.q_pop[qi], ((u64)t << 32) | (u32)(head + 1));
    v.n_del++;
    v.changed = true;
    if (head + 1 != tail) v.nxt = min(v.nxt, t + 1);
    if (!pk_last(pk)) return;
    v.nxt = min(v.nxt, t + 1);                         // DAG looks at its counts next tick
    rank_poke(v, rank_item(*v.X, P.node_rank[v.W->node_off + pk.z]), t + 1);   // the ACK
    u32 ps = pk_slot(pk);
    uint2 port = __ldcg(&P.ports[v.rk * kNPort + ps]);
    port.x++;
    __stcg(&P.ports[v.rk * kNPort + ps], port);
    u64 own = v.X->nd_off + port.y, snd = v.X->nd_off + pk.z;
    atomicMax(&P.nd_done[own], t);
    __threadfence();
    atomicSub(&P.nd_out[own], 1);
    atomicMax(&P.nd_done[snd], t + pk_hops(pk));
    __threadfence();
    atomicSub(&P.nd_out[snd], 1);
    v.n_msg++;
    v.dig += mix64(mix64((u64)pk.z | ((u64)pk_key(pk) << 32)) ^ (u64)t);
    if (v.X->rec_cap) {
        u32 idx = atomicAdd(&v.c->rec_count, 1);
        if (idx < v.X->rec_cap) {
            P.rec_sender[v.X->rec_off + idx] = pk.z;
            P.rec_key[v.X->rec_off + idx] = pk_key(pk);
            P.rec_tick[v.X->rec_off + idx] = t;
        }
    } else {
        atomicAdd(&v.c->rec_count, 1);
    }
}

__device__ __noinline__ void rank_tick(const Params &P, const ExpRec &X, u32 e, u32 r, u32 t, u32 k)
{
    const TopoRec T = P.topo[X.topo];
    const WorkRec W = P.work[X.work];
    RankView v;
    v.P = &P; v.X = &X; v.T = &T; v.W = &W; v.c = &P.ctl[e];
    v.r = r; v.t = t; v.e = e; v.k = k; v.rk = X.rk_off + r;
    v.changed = v.fail_over = v.fail_err = false;
    v.nxt = kUnset;
    v.pk_min = kUnset;
    const u32 it = rank_item(X, r - (r % 32));
    u32 old = 0;
    if ((threadIdx.x & 31) == 0) old = atomicExch(&P.wake[it], kUnset);
    old = __shfl_sync(0xffffffffu, old, 0);
    v.n_inj = v.n_del = v.n_msg = v.n_done = v.end_max1 = 0;
    v.dig = 0;
    const bool active = r < X.nr;
    if (active) {
        v.C = load_ctl(&P.rk[v.rk]);
        dag_step(v);
        if (!v.fail_over && !v.fail_err) {
            inject(v);
            receive(v);
        }
        store_ctl(&P.rk[v.rk], v.C);
    }
    const u32 full = 0xffffffffu;
    u32 nxt = __reduce_min_sync(full, v.nxt);
    u32 pkm = __reduce_min_sync(full, v.pk_min);
    u32 inj = __reduce_add_sync(full, v.n_inj);
    u32 del = __reduce_add_sync(full, v.n_del);
    u32 msg = __reduce_add_sync(full, v.n_msg);
    u32 done = __reduce_add_sync(full, v.n_done);
    u32 emax = __reduce_max_sync(full, v.end_max1);
    bool over = __any_sync(full, v.fail_over), err = __any_sync(full, v.fail_err);
    // 64-bit digest sum across the warp
    u64 dig = v.dig;
    for (int o = 16; o > 0; o >>= 1) dig += __shfl_xor_sync(full, dig, o);
    if ((threadIdx.x & 31) == 0) {
        ExpCtl *c = v.c;
        u32 w = min(nxt, old > t ? old : kUnset);
        if (w != kUnset) atomicMin(&P.wake[it], w);
        u32 m = min(w, pkm);
        if (m != kUnset) atomicMin(&c->nxt[k % 3], m);
        if (inj) {
            atomicAdd((unsigned long long *)&c->pkts_injected, (unsigned long long)inj);
            atomicAdd((unsigned long long *)&c->pkt_hops, (unsigned long long)inj);
        }
        if (del) atomicAdd((unsigned long long *)&c->pkts_delivered, (unsigned long long)del);
        if (msg) {
            atomicAdd((unsigned long long *)&c->msgs_delivered, (unsigned long long)msg);
            atomicAdd((unsigned long long *)&c->digest, (unsigned long long)dig);
        }
        if (emax) atomicMax(&c->end_max1, emax);
        if (done && atomicSub(&c->nodes_left, done) == done) atomicMin(&c->stop_step, k);
        if (over) set_status(c, EXP_OVERFLOW, k);
        if (err) set_status(c, EXP_ERROR, k);
    }
}

// ---------------------------------------------------------------- megakernel
constexpr int kBlock = 512;
constexpr int kWarps = kBlock / 32;

// Each warp owns a contiguous chunk of work items (an experiment's items are
// contiguous: its switches, then its rank groups).  Per step it reads the
// wake ticks of 32 items at once, ballots the ones due, reports the pending
// wakes of the others (one atomic per experiment per warp), and processes the
// due ones one after the other with the whole warp.
__global__ void __launch_bounds__(kBlock, 1) k_megakernel(Params P)
{
    __shared__ SwSmem smem[kWarps];
    const u32 full = 0xffffffffu;
    const u32 warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const u32 gwarp = blockIdx.x * kWarps + warp;
    const u32 nwarps = gridDim.x * kWarps;
    const u32 per = (P.n_items + nwarps - 1) / nwarps;
    const u32 i0 = min(gwarp * per, P.n_items), i1 = min(i0 + per, P.n_items);
    const bool leader_thread = blockIdx.x == 0 && threadIdx.x == 0;
    for (u32 k = 0;; k++) {
        if (leader_thread) P.glob->run_cnt[(k + 1) % 3] = 0;   // last read after barrier k-2
        for (u32 base = i0; base < i1; base += 32) {
            const u32 it = base + lane;
            const bool valid = it < i1;
            const u32 e = valid ? P.item_exp[it] : kUnset;
            const u32 loc = valid ? P.item_loc[it] : 0;
            const u32 t = valid ? exp_tick(P, e, k) : kUnset;
            if (valid && loc == 0) exp_control(P, e, k, t);
            const u32 w = t != kUnset ? ld_rlx32(&P.wake[it]) : kUnset;
            const bool due = t != kUnset && w <= t;
            const u32 peers = __match_any_sync(full, e);
            const u32 rep = __reduce_min_sync(peers, due ? kUnset : w);
            if (e != kUnset && rep != kUnset && lane == (u32)__ffs(peers) - 1)
                atomicMin(&P.ctl[e].nxt[k % 3], rep);
            u32 M = __ballot_sync(full, due);
            while (M) {
                const u32 j = (u32)__ffs(M) - 1;
                M &= M - 1;
                const u32 ej = __shfl_sync(full, e, j), lj = __shfl_sync(full, loc, j),
                          tj = __shfl_sync(full, t, j);
                const ExpRec X = P.exp[ej];
                if (lj < X.nsw) switch_tick(P, X, ej, lj, tj, k, &smem[warp]);
                else rank_tick(P, X, ej, (lj - X.nsw) * 32 + lane, tj, k);
            }
        }
        if (!grid_barrier(P, k)) break;
        if (ld_rlx32(&P.glob->run_cnt[k % 3]) == 0) {
            if (leader_thread) P.glob->steps = k + 1;
            break;
        }
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
    k_up_lists<<<blocks ? (blocks > 1024 ? 1024 : blocks) : 1, 256, 0, st>>>(p, n_sw_total);
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
    dim3 grid(bx, p.n_exps);
    k_init<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_run_reset(const Params &p, u32 max_ticks, cudaStream_t st)
{
    u32 blocks = (p.n_exps + 255) / 256;
    k_run_reset<<<blocks ? blocks : 1, 256, 0, st>>>(p, max_ticks);
    return cudaGetLastError();
}

cudaError_t megakernel_occupancy(int *blocks_per_sm, int *n_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_megakernel, kBlock, 0);
}

cudaError_t launch_megakernel(const Params &p, u32 blocks, cudaStream_t st)
{
    Params q = p;
    void *args[] = {&q};
    return cudaLaunchCooperativeKernel((void *)k_megakernel, dim3(blocks), dim3(kBlock), args, 0,
                                       st);
}

}  // namespace mv
