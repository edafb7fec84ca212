/*
 * mv_oracle.c -- plain, slow, single-threaded CPU oracle for the lock-step
 * packet simulation of collective traffic.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header or table with the CUDA library; both read the same flat batch
 * arrays produced by the seeded input generators.
 *
 * What it follows (page = "Accelerating Design Space Exploration for LLM
 * Training Systems with Multi-experiment Parallel Simulation", Multiverse):
 *   - section 3.2, "system execution graph": one simulation step runs, in
 *     order, Schedule/AnalyticalSys (DAG advance), the switch forwarding
 *     systems, NIC send and NIC receive/ACK.  Here one step is one tick.
 *   - section 4.2: forwarding is split into a per-ingress plan (which egress
 *     the head packet wants) and a per-egress pull from the ingress ports.
 *   - section 4.1: intra-server collectives take alpha + bytes/beta.
 *   - section 3.1: the GPU memory check runs before the simulation.
 *   - section 5: ring all-reduce / all-gather / reduce-scatter, ECMP.
 * and from "AutoCCL" section 2.3: a message is split into NC partitions, one
 * per channel, each cut into chunks of C bytes; from "On Optimizing the
 * Communication of Model Parallelism" section 3.1: the pipelined broadcast
 * in which each receiver forwards a partition once it holds it whole.
 *
 * Every experiment is simulated on its own, tick by tick, with one object
 * per entity.  Within a tick the phases run over all entities in index
 * order.  Information that crosses entities is never from the current tick:
 * queue entries become visible at their ready tick, credit for a popped
 * entry travels back over its link (delta + 1 ticks), a rank's join reaches
 * its peers after one minimum link latency, and acknowledgements carry their
 * own arrival tick.  That makes the result independent of the order entities
 * are visited in.
 *
 * Parity pins live in tests/: the lone-message and heterogeneous-path closed
 * forms, the pipelined broadcast closed form, a contention-free ring
 * evaluated as a longest path, hand-traced tick tables (matched event by
 * event through the trace below), schedule details derived by hand (ring
 * blocks, lane round robin, partitions, all-to-all striping, tree
 * children), DAG critical paths, the analytic model, the memory check, the
 * table and tick limits, idle-tick skipping against stepping every tick,
 * and the run-time invariant counts; a mutation test plants plausible
 * mistakes here and requires those pins to fail.  Parity unpinned: which
 * up port the ECMP hash gives a particular connection (route_port) is this
 * build's convention; the pins fix only its properties (one path per
 * connection, spread over the up ports, dependence on seed and switch).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define UNSET 0xFFFFFFFFu
#define NLANE 64      /* send lanes per NIC (active messages streams)   */
#define NPORT 128     /* receive counters per rank                      */
#define NPTAB 64      /* notification-point flow table entries per NIC  */
#define NCNPQ 64      /* control packets waiting at a NIC (DCQCN uses 16) */
#define NPEND 64      /* scheduled-but-not-started nodes per rank       */
#define NACT 16       /* running collective memberships per rank        */
#define TICK_LIMIT 0xFFF00000u   /* largest tick value a run reaches        */

enum { K_COMPUTE = 0, K_INTRA = 1, K_NET = 2 };
enum { C_AR = 0, C_RS = 1, C_AG = 2, C_RELAY = 3, C_P2P = 4, C_A2A = 5 };
enum { A_RING = 0, A_TREE = 1 };
enum { ST_DONE = 0, ST_RUNNING = 1, ST_OOM = 2, ST_DEADLOCK = 3, ST_OVERFLOW = 4,
       ST_ERROR = 5 };

typedef struct orc_batch {
    uint32_t version;
    uint32_t n_topos, n_works, n_exps;
    const uint32_t *topo_nhosts, *topo_nsw, *topo_nports;
    const uint32_t *sw_nports, *sw_level;
    const int32_t *port_peer;
    const uint32_t *port_sigma, *port_delta, *host_port, *host_sigma, *host_delta;
    const uint32_t *work_nranks, *work_nnodes, *work_nedges, *work_ncolls,
        *work_nmembers, *work_na2a, *work_na2a_in;
    const uint32_t *rank_nnodes, *node_kind, *node_arg, *node_npred, *node_nsucc,
        *node_dur_lo, *node_dur_hi, *node_dur_key, *succ;
    const uint32_t *coll_kind, *coll_intra;
    const uint64_t *coll_bytes;
    const uint32_t *coll_nmembers, *coll_parts, *coll_alpha, *coll_beta_num,
        *coll_beta_den, *member_rank, *member_node, *member_a2a_n, *a2a_dst;
    const uint64_t *a2a_bytes;
    const uint32_t *member_a2a_in_n, *a2a_in_src;
    const uint64_t *a2a_in_bytes;
    const uint64_t *mem;
    const uint32_t *exp_topo, *exp_work, *exp_algo, *exp_nc;
    const uint64_t *exp_chunk;
    const uint32_t *exp_pkt, *exp_cap, *exp_tick_ps;
    const uint64_t *exp_dur_seed, *exp_ecmp_seed, *exp_gpu_mem;
    const uint32_t *exp_rec_cap;
    const uint32_t *exp_voq;
    const uint32_t *exp_cc;       /* n_exps x CC_FIELDS; NULL: no congestion control */
} orc_batch;

typedef struct orc_out {
    uint32_t *status, *end_tick, *now;
    uint64_t *pkts_injected, *pkt_hops, *pkts_delivered, *msgs_delivered, *digest,
        *ticks_active;
    uint32_t *node_start, *node_end;        /* concatenated per experiment */
    uint32_t *rec_count;                    /* per experiment */
    uint32_t *rec_sender, *rec_key, *rec_tick; /* concatenated, rec_cap each */
    uint64_t *violations;                   /* per experiment: broken invariants */
    /* per collective instance, concatenated per experiment (the workload's
     * collectives in order): earliest member start and latest member end;
     * UNSET while some member has not ended (optional: may be NULL) */
    uint32_t *coll_start, *coll_end;
} orc_out;

/* Optional event trace of one run (parity bisection): what happened at which
 * tick, in the order the serial phases meet it.
 *   EV_START   a = node, b = rank          EV_END     a = node, b = end tick
 *   EV_INJECT  a = rank, b = connection key
 *   EV_HOP     a = egress port, b = ingress queue it pulled from (switch hop)
 *   EV_DELIVER a = rank, b = sender node   EV_MESSAGE a = rank, b = sender node
 *                                            (the message's last packet) */
typedef struct orc_event {
    uint32_t tick, kind, a, b;
} orc_event;
enum { EV_START = 1, EV_END = 2, EV_INJECT = 3, EV_HOP = 4, EV_DELIVER = 5, EV_MESSAGE = 6,
       EV_CNP = 7, EV_CUT = 8, EV_WINDOW = 9, EV_ACK = 10 };

/* Congestion control of an experiment (CC_FIELDS words each).  CC_ON: 0
 * none, 1 DCQCN, 2 DCTCP.  DCQCN: switch marking thresholds in packets and
 * the marking probability at kmax (units of 2^-16); the gain g = 2^-gshift;
 * the notification gap N, the alpha timer K and the rate timer T in ticks;
 * the byte counter B in packets; the fast recovery count F; the additive,
 * hyper and minimum rates in units of 2^-20 of the line rate.  DCTCP: the
 * marking threshold (kmin = kmax), the gain shift, and the initial and
 * largest window in packets (CC_W0, CC_WMAX). */
enum { CC_ON, CC_KMIN, CC_KMAX, CC_PMAX, CC_GSHIFT, CC_N, CC_K, CC_T, CC_B, CC_F, CC_RAI,
       CC_RHAI, CC_RMIN, CC_W0, CC_WMAX, CC_FIELDS = 16 };
enum { CC_DCQCN = 1, CC_DCTCP = 2 };
#define CC_LINE (1u << 20)        /* the line rate in rate units */
#define ORC_NO_SKIP 1u

/* ------------------------------------------------------------------------ */
/* splitmix64 finaliser (S. Vigna, public domain splitmix64.c): the one
 * counter-based hash used for ECMP, durations and the digest.              */
static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t umin(uint64_t a, uint64_t b) { return a < b ? a : b; }
static uint32_t umax32(uint32_t a, uint32_t b) { return a > b ? a : b; }

/* ------------------------------------------------------------------------ */
typedef struct pkt {
    uint32_t ready, dst, hopsum, sender, pslot, last, key;
    uint32_t lane, ecn;           /* the sender's lane slot; congestion experienced */
    uint32_t cnp;                 /* a control packet for lane `lane` of host dst: a DCQCN
                                     notification, or a DCTCP acknowledgement of n packets,
                                     m of them marked */
    uint32_t n, m;
} pkt;

typedef struct lane {
    int used;
    uint32_t node, member, chan, kind;
    uint32_t m, nmsg, pkts_left;
    uint32_t dst_member, dst_port, dep_base, dep_mask, dep_need, key;
    uint32_t a2a_e, a2a_start;
    /* DCQCN reaction point: current and target rate, alpha, the earliest
     * tick of the next packet, the alpha and rate timers' last expiry, the
     * rate timer and byte counter event counts, and packets since the last
     * byte-counter event */
    uint32_t rc, rt, alpha, next_tx, abase, rbase, tc, bc, sent;
    /* DCTCP sender: window (units of 2^-10 packets), packets sent and
     * acknowledged, the acknowledged count that closes the observation
     * window, acknowledgements and marks in it; a lane that sent all its
     * messages keeps its slot (draining) until every packet is acknowledged */
    uint32_t wnd, sentc, acked, wend, wa, wm, draining;
} lane;

typedef struct nic {
    uint32_t busy, rr;
    lane lanes[NLANE];
    int port_used[NPORT];
    uint32_t port_count[NPORT];
    uint32_t port_node[NPORT];
    uint32_t pend_node[NPEND], pend_start[NPEND];
    int n_pend;
    int n_lanes;          /* lanes in use (skip the scan when none)        */
    uint64_t used_mask;   /* bit q set when lane slot q is in use           */
    uint32_t act[NACT];
    int n_act;
    int tick_fail;        /* one of its tables overflowed during this tick  */
    /* DCQCN notification point: the last notification generated per flow,
     * in a direct-mapped table (flow key mod NPTAB), and the notifications
     * waiting to be sent (a ring of NCNPQ) */
    uint32_t np_key[NPTAB], np_at[NPTAB];
    uint32_t cq_dst[NCNPQ], cq_lane[NCNPQ], cq_key[NCNPQ], cq_n[NCNPQ], cq_m[NCNPQ], cq_head,
        cq_tail;
} nic;

typedef struct sim {
    const orc_batch *b;
    uint32_t e;
    /* topology views (topology-local indices) */
    uint32_t H, S, Q;
    const uint32_t *sw_nports, *sw_level, *port_sigma, *port_delta, *host_port,
        *host_sigma, *host_delta;
    const int32_t *port_peer;
    uint32_t *sw_base;     /* S+1 */
    uint32_t *port_sw;     /* Q   */
    int32_t *route;        /* S*H: down port (switch-local) or -1 */
    uint32_t *up_base, *up_port;
    /* workload views (workload-local indices) */
    uint32_t R, NN;
    uint32_t *rank_base;   /* R+1 */
    uint32_t *node_rank;   /* NN */
    uint32_t *succ_base;   /* NN+1 */
    uint32_t *member_base; /* ncolls+1 */
    uint32_t *row_base, *col_base; /* nmembers+1 */
    uint32_t *node_member; /* NN: member index for collective nodes */
    const uint32_t *node_kind, *node_arg, *node_npred, *node_dur_lo, *node_dur_hi,
        *node_dur_key, *succ, *coll_kind, *coll_intra, *coll_nmembers, *coll_parts,
        *coll_alpha, *coll_beta_num, *coll_beta_den, *member_rank, *member_node,
        *a2a_dst, *a2a_in_src;
    const uint64_t *coll_bytes, *a2a_bytes, *a2a_in_bytes, *mem;
    /* experiment parameters */
    uint32_t algo, nc, pkt, cap, tick_ps, rec_cap;
    uint64_t chunk, dur_seed, ecmp_seed, gpu_mem;
    /* dynamic state */
    uint32_t nf;                    /* queues: Q switch ingress + H NIC rx */
    uint32_t *head, *tail, *tail0;
    uint32_t *poplog;               /* nf * 64: tick of each of the last 64 pops */
    uint32_t *credit_delay;         /* nf: delta + 1 of the link feeding the queue */
    uint32_t rdv_delay;             /* 1 + smallest link delta of the topology */
    pkt *slots;                     /* nf * cap */
    uint32_t *eg_busy, *eg_rr;      /* Q */
    int voq;                        /* switches keep virtual output queues */
    uint32_t cc[CC_FIELDS];         /* DCQCN parameters (cc[CC_ON] = 0: none) */
    uint64_t *taken;                /* Q: with VOQs, ring slots already forwarded (by slot) */
    uint32_t *sw_queued;            /* S: packets in the switch's ingress queues */
    nic *nics;                      /* R */
    uint32_t *npred_left, *cand, *start, *end, *port_base, *done_max;
    int64_t *outstanding;
    uint32_t nodes_left;
    int changed, status;
    int cur_rank;                   /* rank whose DAG step is running, or -1 */
    uint64_t pkts_injected, pkt_hops, pkts_delivered, msgs_delivered, digest;
    uint32_t *rec_sender, *rec_key, *rec_tick, rec_count;
    /* invariant checks, independent of the state that enforces them: a
     * queue never holds more than cap packets; the one link feeding a queue
     * carries at most one packet per its serialisation time; a packet is
     * delivered at the host it was addressed to */
    uint32_t *last_push;            /* nf: tick of the last push into the queue */
    uint64_t violations;
    /* event trace (none when trace is NULL): events beyond trace_cap are
     * counted, not kept */
    orc_event *trace;
    uint64_t trace_cap, trace_n;
    uint32_t now;                   /* the tick being simulated */
    int no_skip;                    /* step every tick instead of jumping to the next event */
    uint32_t t_next;                /* the next tick to simulate (a paused run resumes here) */
    uint64_t active;                /* ticks simulated so far */
    int is_clone;                   /* shares the read-only tables of the sim it was copied from */
} sim;

static void ev(sim *s, uint32_t kind, uint32_t a, uint32_t b)
{
    if (!s->trace) return;
    if (s->trace_n < s->trace_cap) {
        orc_event *x = &s->trace[s->trace_n];
        x->tick = s->now;
        x->kind = kind;
        x->a = a;
        x->b = b;
    }
    s->trace_n++;
}

/* A failure stops the experiment at the end of the current tick.  Within
 * that tick every other entity still completes its step (Multiverse section
 * 3.2: a system processes all of its entities in one invocation), while the
 * rank that failed does nothing more.  The first failure in the phase order
 * (ranks in index order, then switches) names the status. */
static void fail(sim *s, int st)
{
    if (s->status == ST_RUNNING) s->status = st;
    if (s->cur_rank >= 0) s->nics[s->cur_rank].tick_fail = 1;
}

/* ------------------------------------------------------------------------ */
/* Routing: shortest up/down.  A switch forwards down when the destination
 * host sits below one of its down ports (the lowest such port), otherwise up
 * on a port chosen by the per-connection ECMP hash (Multiverse section 5).   */
static void build_routes(sim *s)
{
    uint32_t S = s->S, H = s->H;
    s->route = malloc(sizeof(int32_t) * (size_t)S * H);
    for (size_t i = 0; i < (size_t)S * H; i++) s->route[i] = -1;
    uint32_t maxlev = 0;
    for (uint32_t w = 0; w < S; w++) maxlev = umax32(maxlev, s->sw_level[w]);
    for (uint32_t lev = 1; lev <= maxlev; lev++) {
        for (uint32_t w = 0; w < S; w++) {
            if (s->sw_level[w] != lev) continue;
            for (uint32_t p = 0; p < s->sw_nports[w]; p++) {
                int32_t pe = s->port_peer[s->sw_base[w] + p];
                if (pe < 0) {
                    uint32_t h = (uint32_t)(-pe - 1);
                    if (s->route[(size_t)w * H + h] < 0) s->route[(size_t)w * H + h] = (int32_t)p;
                } else {
                    uint32_t w2 = s->port_sw[pe];
                    if (s->sw_level[w2] >= lev) continue;
                    for (uint32_t h = 0; h < H; h++)
                        if (s->route[(size_t)w2 * H + h] >= 0 && s->route[(size_t)w * H + h] < 0)
                            s->route[(size_t)w * H + h] = (int32_t)p;
                }
            }
        }
    }
    s->up_base = calloc(S + 1, sizeof(uint32_t));
    s->up_port = malloc(sizeof(uint32_t) * (s->Q + 1));
    uint32_t k = 0;
    for (uint32_t w = 0; w < S; w++) {
        s->up_base[w] = k;
        for (uint32_t p = 0; p < s->sw_nports[w]; p++) {
            int32_t pe = s->port_peer[s->sw_base[w] + p];
            if (pe >= 0 && s->sw_level[s->port_sw[pe]] > s->sw_level[w]) s->up_port[k++] = p;
        }
    }
    s->up_base[S] = k;
}

/* egress port (switch-local) for a packet at switch w.  Parity unpinned for
 * the exact up port the hash picks (a convention); see the header. */
static int32_t route_port(sim *s, uint32_t w, const pkt *p)
{
    int32_t d = s->route[(size_t)w * s->H + p->dst];
    if (d >= 0) return d;
    uint32_t nup = s->up_base[w + 1] - s->up_base[w];
    if (nup == 0) return -1;
    uint64_t h = mix64((uint64_t)p->key ^ ((uint64_t)w << 40) ^ s->ecmp_seed);
    return (int32_t)s->up_port[s->up_base[w] + (uint32_t)(h % nup)];
}

/* ------------------------------------------------------------------------ */
/* Collective decomposition into messages (AutoCCL section 2.3 for NC and C;
 * the ring schedule of NCCL named on the Multiverse page, section 5).       */
static uint32_t coll_of(sim *s, uint32_t node) { return s->node_arg[node]; }
static uint32_t nmemb(sim *s, uint32_t c) { return s->coll_nmembers[c]; }
static uint32_t mrank(sim *s, uint32_t c, uint32_t i) { return s->member_rank[s->member_base[c] + i]; }
static uint32_t mnode(sim *s, uint32_t c, uint32_t i) { return s->member_node[s->member_base[c] + i]; }

static int is_tree(sim *s, uint32_t c) { return s->coll_kind[c] == C_AR && s->algo == A_TREE; }

static uint32_t n_chan(sim *s, uint32_t c)
{
    uint32_t k = s->coll_kind[c];
    return (k == C_RELAY || k == C_P2P) ? 1 : s->nc;
}
/* lanes per channel / ports per channel */
static uint32_t lanes_per_chan(sim *s, uint32_t c) { return is_tree(s, c) ? 3 : 1; }
static uint32_t n_ports(sim *s, uint32_t c)
{
    uint32_t k = s->coll_kind[c];
    if (k == C_RELAY || k == C_P2P || k == C_A2A) return 1;
    return n_chan(s, c) * (is_tree(s, c) ? 3 : 1);
}

/* bytes of channel c's partition: the first S mod NC partitions get one more */
static uint64_t partition(uint64_t S, uint32_t nc, uint32_t c)
{
    return S / nc + (c < S % nc ? 1 : 0);
}

static uint32_t ring_steps(sim *s, uint32_t c)
{
    uint32_t N = nmemb(s, c);
    if (N < 2) return 0;
    return s->coll_kind[c] == C_AR ? 2 * (N - 1) : N - 1;
}

static uint64_t ring_loops(sim *s, uint32_t c, uint64_t P)
{
    uint64_t stride = (uint64_t)nmemb(s, c) * s->chunk;
    return P == 0 ? 1 : ceil_div(P, stride);
}

static uint64_t n_chunks(uint64_t bytes, uint64_t C) { return bytes == 0 ? 1 : ceil_div(bytes, C); }

/* number of messages lane (chan, kind) of member i sends */
static uint32_t lane_nmsg(sim *s, uint32_t c, uint32_t i, uint32_t chan, uint32_t kind)
{
    uint32_t N = nmemb(s, c);
    uint64_t S = s->coll_bytes[c];
    switch (s->coll_kind[c]) {
    case C_AR: case C_RS: case C_AG:
        if (is_tree(s, c)) {
            uint64_t nch = n_chunks(partition(S, s->nc, chan), s->chunk);
            if (kind == 0) return i > 0 ? (uint32_t)nch : 0;
            if (kind == 1) return 2 * i + 1 < N ? (uint32_t)nch : 0;
            return 2 * i + 2 < N ? (uint32_t)nch : 0;
        }
        return (uint32_t)(ring_loops(s, c, partition(S, s->nc, chan)) * ring_steps(s, c));
    case C_RELAY:
        return i + 1 < N ? s->coll_parts[c] : 0;
    case C_P2P:
        return i == 0 ? (uint32_t)n_chunks(S, s->chunk) : 0;
    case C_A2A: {
        uint64_t tot = 0;
        for (uint32_t e = s->row_base[s->member_base[c] + i]; e < s->row_base[s->member_base[c] + i + 1]; e++)
            tot += n_chunks(s->a2a_bytes[e], s->chunk);
        return tot > chan ? (uint32_t)ceil_div(tot - chan, s->nc) : 0;
    }
    }
    return 0;
}

/* messages expected on receive port p of member i */
static uint32_t port_expect(sim *s, uint32_t c, uint32_t i, uint32_t p)
{
    uint32_t N = nmemb(s, c);
    uint64_t S = s->coll_bytes[c];
    switch (s->coll_kind[c]) {
    case C_AR: case C_RS: case C_AG:
        if (is_tree(s, c)) {
            uint32_t chan = p / 3, q = p % 3;
            uint64_t nch = n_chunks(partition(S, s->nc, chan), s->chunk);
            if (q == 0) return i > 0 ? (uint32_t)nch : 0;
            if (q == 1) return 2 * i + 1 < N ? (uint32_t)nch : 0;
            return 2 * i + 2 < N ? (uint32_t)nch : 0;
        }
        return (uint32_t)(ring_loops(s, c, partition(S, s->nc, p)) * ring_steps(s, c));
    case C_RELAY:
        return i > 0 ? s->coll_parts[c] : 0;
    case C_P2P:
        return i == 1 ? (uint32_t)n_chunks(S, s->chunk) : 0;
    case C_A2A: {
        uint64_t tot = 0;
        for (uint32_t e = s->col_base[s->member_base[c] + i]; e < s->col_base[s->member_base[c] + i + 1]; e++)
            tot += n_chunks(s->a2a_in_bytes[e], s->chunk);
        return (uint32_t)tot;
    }
    }
    return 0;
}

/* Fill in message m of a lane: its bytes, destination, destination port and
 * the receive counts it waits for.  Returns the packet count. */
static uint32_t lane_setup(sim *s, lane *L)
{
    uint32_t c = coll_of(s, L->node);
    uint32_t N = nmemb(s, c), i = L->member, m = L->m, chan = L->chan;
    uint64_t S = s->coll_bytes[c], C = s->chunk, bytes = 0;
    L->dep_mask = 0;
    L->dep_need = 0;
    L->dep_base = 0;
    switch (s->coll_kind[c]) {
    case C_AR: case C_RS: case C_AG: {
        uint64_t P = partition(S, s->nc, chan);
        if (is_tree(s, c)) {
            uint32_t has_l = 2 * i + 1 < N, has_r = 2 * i + 2 < N;
            bytes = P > (uint64_t)m * C ? umin(C, P - (uint64_t)m * C) : 0;
            uint32_t child_mask = (has_l ? 2u : 0u) | (has_r ? 4u : 0u);
            if (L->kind == 0) {               /* reduce: up to the parent */
                uint32_t par = (i - 1) / 2;
                L->dst_member = par;
                L->dst_port = chan * 3 + (i == 2 * par + 1 ? 1 : 2);
                L->dep_mask = child_mask;
            } else {                          /* broadcast: down to a child */
                L->dst_member = 2 * i + L->kind;
                L->dst_port = chan * 3;
                L->dep_mask = i == 0 ? child_mask : 1u;
            }
            L->dep_need = m + 1;
            L->dep_base = chan * 3;
        } else {
            uint32_t steps = ring_steps(s, c);
            uint64_t l = m / steps, k = m % steps;
            uint64_t stride = (uint64_t)N * C;
            uint64_t B = umin(stride, P - l * stride);
            uint64_t bs = ceil_div(B, N);
            uint64_t blk = ((uint64_t)i + N - (k % N)) % N;   /* (i - k) mod N */
            bytes = B > blk * bs ? umin(bs, B - blk * bs) : 0;
            L->dst_member = (i + 1) % N;
            L->dst_port = chan;
            L->dep_base = chan;
            if (k >= 1) { L->dep_mask = 1u; L->dep_need = (uint32_t)(l * steps + k); }
        }
        break;
    }
    case C_RELAY: {
        uint32_t K = s->coll_parts[c];
        bytes = S / K + (m < S % K ? 1 : 0);
        L->dst_member = i + 1;
        L->dst_port = 0;
        if (i >= 1) { L->dep_mask = 1u; L->dep_need = m + 1; }
        break;
    }
    case C_P2P:
        bytes = S > (uint64_t)m * C ? umin(C, S - (uint64_t)m * C) : 0;
        L->dst_member = 1;
        L->dst_port = 0;
        break;
    case C_A2A: {
        uint32_t r0 = s->row_base[s->member_base[c] + i];
        uint64_t g = (uint64_t)chan + (uint64_t)m * s->nc;
        while (g >= L->a2a_start + n_chunks(s->a2a_bytes[r0 + L->a2a_e], C)) {
            L->a2a_start += (uint32_t)n_chunks(s->a2a_bytes[r0 + L->a2a_e], C);
            L->a2a_e++;
        }
        uint64_t j = g - L->a2a_start, b = s->a2a_bytes[r0 + L->a2a_e];
        bytes = b > j * C ? umin(C, b - j * C) : 0;
        L->dst_member = s->a2a_dst[r0 + L->a2a_e];
        L->dst_port = 0;
        break;
    }
    }
    uint32_t drank = mrank(s, c, L->dst_member);
    L->key = (uint32_t)(mix64((uint64_t)L->node | ((uint64_t)(chan * 4 + L->kind) << 32) |
                              ((uint64_t)drank << 44)) & 0xFFFFFFu);
    return (uint32_t)(bytes == 0 ? 1 : ceil_div(bytes, s->pkt));
}

/* ------------------------------------------------------------------------ */
/* DAG advance (Schedule + AnalyticalSys, Multiverse section 3.2)           */
static uint32_t compute_ticks(sim *s, uint32_t u)
{
    uint64_t lo = s->node_dur_lo[u], hi = s->node_dur_hi[u], ns = lo;
    if (hi > lo) ns = lo + mix64(mix64((uint64_t)s->node_dur_key[u]) ^ s->dur_seed) % (hi - lo + 1);
    return (uint32_t)ceil_div(ns * 1000, s->tick_ps);
}

/* Analytic intra-server time (Multiverse section 4.1): alpha + bytes/beta
 * with beta given as ticks per byte beta_num/beta_den, and the bytes each
 * GPU moves: 2(g-1)S/g for all-reduce, (g-1)S/g for all-gather and
 * reduce-scatter, S otherwise. */
static uint32_t intra_ticks(sim *s, uint32_t c)
{
    uint64_t g = nmemb(s, c), S = s->coll_bytes[c], be;
    switch (s->coll_kind[c]) {
    case C_AR: be = ceil_div(2 * (g - 1) * S, g); break;
    case C_RS: case C_AG: be = ceil_div((g - 1) * S, g); break;
    default: be = S;
    }
    return s->coll_alpha[c] + (uint32_t)ceil_div(be * s->coll_beta_num[c], s->coll_beta_den[c]);
}

static void pend_add(sim *s, uint32_t r, uint32_t u, uint32_t st)
{
    nic *n = &s->nics[r];
    if (n->n_pend >= NPEND) { fail(s, ST_OVERFLOW); return; }
    n->pend_node[n->n_pend] = u;
    n->pend_start[n->n_pend] = st;
    n->n_pend++;
}

static void complete(sim *s, uint32_t u, uint32_t c)
{
    ev(s, EV_END, u, c);
    uint32_t r = s->node_rank[u];
    s->end[u] = c;
    s->nodes_left--;
    s->changed = 1;
    if (c >= TICK_LIMIT) { fail(s, ST_OVERFLOW); return; }
    for (uint32_t k = s->succ_base[u]; k < s->succ_base[u + 1]; k++) {
        uint32_t v = s->succ[k];
        s->cand[v] = umax32(s->cand[v], c + 1);
        if (--s->npred_left[v] == 0) pend_add(s, r, v, s->cand[v]);
    }
}

/* a rank joins a network collective: receive counters and send lanes */
static void net_join(sim *s, uint32_t r, uint32_t u, uint32_t t)
{
    nic *n = &s->nics[r];
    uint32_t c = coll_of(s, u), i = s->node_member[u];
    uint32_t np = n_ports(s, c);
    int base = -1;
    for (uint32_t b = 0; b + np <= NPORT && base < 0; b++) {
        uint32_t k = 0;
        while (k < np && !n->port_used[b + k]) k++;
        if (k == np) base = (int)b;
    }
    if (base < 0) { fail(s, ST_OVERFLOW); return; }
    int64_t out = 0;
    for (uint32_t p = 0; p < np; p++) {
        n->port_used[base + p] = 1;
        n->port_count[base + p] = 0;
        n->port_node[base + p] = u;
        out += port_expect(s, c, i, p);
    }
    s->port_base[u] = (uint32_t)base;
    uint32_t nch = n_chan(s, c), lpc = lanes_per_chan(s, c);
    for (uint32_t ch = 0; ch < nch; ch++) {
        for (uint32_t k = 0; k < lpc; k++) {
            uint32_t nm = lane_nmsg(s, c, i, ch, k);
            if (nm == 0) continue;
            int slot = -1;
            for (int q = 0; q < NLANE && slot < 0; q++)
                if (!n->lanes[q].used) slot = q;
            if (slot < 0) { fail(s, ST_OVERFLOW); return; }
            lane *L = &n->lanes[slot];
            memset(L, 0, sizeof *L);
            L->used = 1;
            L->node = u; L->member = i; L->chan = ch; L->kind = k;
            L->m = 0; L->nmsg = nm;
            L->rc = L->rt = L->alpha = CC_LINE;
            L->abase = L->rbase = t;
            L->wnd = s->cc[CC_W0] << 10;
            L->wend = s->cc[CC_W0];
            L->pkts_left = lane_setup(s, L);
            n->n_lanes++;
            n->used_mask |= 1ULL << slot;
            out += nm;
        }
    }
    s->outstanding[u] = out;
    s->done_max[u] = t;
}

static void free_ports(sim *s, uint32_t r, uint32_t u)
{
    uint32_t np = n_ports(s, coll_of(s, u));
    for (uint32_t p = 0; p < np; p++) s->nics[r].port_used[s->port_base[u] + p] = 0;
}

static void act_add(sim *s, uint32_t r, uint32_t u)
{
    nic *n = &s->nics[r];
    if (n->n_act >= NACT) { fail(s, ST_OVERFLOW); return; }
    int j = n->n_act++;                   /* insert in node order */
    while (j > 0 && n->act[j - 1] > u) { n->act[j] = n->act[j - 1]; j--; }
    n->act[j] = u;
}

static int cmp_u32(const void *a, const void *b)
{
    uint32_t x = *(const uint32_t *)a, y = *(const uint32_t *)b;
    return x < y ? -1 : x > y;
}

static void dag_step(sim *s, uint32_t r, uint32_t t)
{
    nic *n = &s->nics[r];
    if (n->n_act == 0) {                  /* nothing running: anything due now? */
        int due = 0;
        for (int k = 0; k < n->n_pend && !due; k++) due = n->pend_start[k] <= t;
        if (!due) return;
    }
    /* (a) running collectives, in node order (the list is kept sorted):
     * has this member finished? */
    int nk = 0, na = n->n_act;
    for (int a = 0; a < na; a++) {
        uint32_t u = n->act[a], c = coll_of(s, u);
        int fin = 0;
        if (s->node_kind[u] == K_INTRA) {
            uint32_t N = nmemb(s, c), b = 0, ok = 1;
            for (uint32_t j = 0; j < N && ok; j++) {
                uint32_t st = s->start[mnode(s, c, j)];
                if (st == UNSET || st >= t) ok = 0;
                else b = umax32(b, st);
            }
            if (ok) { complete(s, u, b + intra_ticks(s, c)); fin = 1; }
        } else if (s->outstanding[u] == 0) {
            free_ports(s, r, u);
            complete(s, u, s->done_max[u]);
            fin = 1;
        }
        if (!fin) n->act[nk++] = u;
    }
    n->n_act = nk;
    /* (b) start the nodes scheduled for this tick, in node order */
    uint32_t now_nodes[NPEND];
    int nn = 0, w = 0;
    for (int k = 0; k < n->n_pend; k++) {
        if (n->pend_start[k] < t) { fail(s, ST_ERROR); return; }
        if (n->pend_start[k] == t) now_nodes[nn++] = n->pend_node[k];
        else { n->pend_node[w] = n->pend_node[k]; n->pend_start[w] = n->pend_start[k]; w++; }
    }
    n->n_pend = w;
    qsort(now_nodes, nn, sizeof(uint32_t), cmp_u32);
    for (int k = 0; k < nn; k++) {
        if (n->tick_fail) return;         /* this rank failed: it starts nothing more */
        uint32_t u = now_nodes[k];
        s->changed = 1;
        switch (s->node_kind[u]) {
        case K_COMPUTE:
            s->start[u] = t;
            ev(s, EV_START, u, r);
            complete(s, u, t + compute_ticks(s, u));
            break;
        case K_INTRA:
            s->start[u] = t;
            ev(s, EV_START, u, r);
            act_add(s, r, u);
            break;
        case K_NET:
            net_join(s, r, u, t);
            if (n->tick_fail) return;     /* a join that does not fit never starts */
            s->start[u] = t;
            ev(s, EV_START, u, r);
            if (s->outstanding[u] == 0) {
                free_ports(s, r, u);
                complete(s, u, t);
            } else {
                act_add(s, r, u);
            }
            break;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* queues: ring buffers of cap slots; head/tail are free-running counters   */
static pkt *slot(sim *s, uint32_t f, uint32_t idx) { return &s->slots[(size_t)f * s->cap + idx % s->cap]; }
static uint32_t q_of_host(sim *s, uint32_t h) { return s->Q + h; }
static uint32_t downstream(sim *s, uint32_t q)
{
    int32_t pe = s->port_peer[q];
    return pe >= 0 ? (uint32_t)pe : q_of_host(s, (uint32_t)(-pe - 1));
}
/* credit: may a sender push into queue f this tick?  Entries popped this
 * tick free their slot from the next tick on (start-of-tick snapshot). */
/* Credit (lossless, PFC-like): a sender may push into queue f at tick t only
 * if the queue holds fewer than cap entries as far as the sender knows.  An
 * entry counts from its push until its pop's credit gets back to the sender,
 * which travels back over the link: pop tick + delta + 1 (the queue's
 * credit_delay).  Pops are at most one per tick, so only the last
 * credit_delay - 1 pops can still be on their way. */
static int has_credit(sim *s, uint32_t f, uint32_t t)
{
    uint32_t h = s->head[f], back = 0, d = s->credit_delay[f];
    while (back < h && back < 64) {
        uint32_t pt = s->poplog[(size_t)f * 64 + (h - 1 - back) % 64];
        if (pt + d <= t) break;          /* this pop's credit has arrived */
        back++;
    }
    return s->tail[f] - (h - back) < s->cap;
}

static void pop(sim *s, uint32_t f, uint32_t t)
{
    s->poplog[(size_t)f * 64 + s->head[f] % 64] = t;
    s->head[f]++;
}
/* the head entry, if it was present at the start of the tick and is ready */
static pkt *ready_head(sim *s, uint32_t f, uint32_t t)
{
    if (s->tail0[f] == s->head[f]) return NULL;
    pkt *p = slot(s, f, s->head[f]);
    return p->ready <= t ? p : NULL;
}

/* push a packet sent at tick t over a link of serialisation time sigma */
static void push(sim *s, uint32_t f, const pkt *p, uint32_t t, uint32_t sigma)
{
    if (s->tail[f] - s->head[f] >= s->cap) s->violations++;
    if (s->last_push[f] != UNSET && t < s->last_push[f] + sigma) s->violations++;
    s->last_push[f] = t;
    *slot(s, f, s->tail[f]) = *p;
    s->tail[f]++;
    if (f < s->Q) s->sw_queued[s->port_sw[f]]++;
}

/* ------------------------------------------------------------------------ */
/* DCQCN (Zhu et al., SIGCOMM 2015, an outside source: the Multiverse page
 * only names the algorithm).  Congestion point: the switch is input-queued,
 * so the packets waiting for a congested egress sit in the ingress queues
 * that feed it; a switch marks a packet it forwards when the ingress queue
 * it leaves held more than kmin arrived (ready) packets at the start of the
 * tick, counting the packet itself: with probability
 * pmax (q - kmin) / (kmax - kmin) up to kmax and always above it.  The draw
 * is a counter-based hash of the tick, the flow key, the queue and the
 * experiment's seed. */
static uint32_t head_at_tick_start(sim *s, uint32_t f, uint32_t t)
{
    uint32_t h = s->head[f];
    return (h > 0 && s->poplog[(size_t)f * 64 + (h - 1) % 64] == t) ? h - 1 : h;
}

static uint32_t ecn_mark(sim *s, uint32_t qin, const pkt *p, uint32_t t)
{
    uint32_t q = 0;
    for (uint32_t x = head_at_tick_start(s, qin, t); x != s->tail0[qin]; x++) {
        if (slot(s, qin, x)->ready > t) break;        /* still on the wire */
        q++;
    }
    if (q <= s->cc[CC_KMIN]) return 0;
    if (q > s->cc[CC_KMAX]) return 1;
    uint64_t prob = (uint64_t)s->cc[CC_PMAX] * (q - s->cc[CC_KMIN]) /
                    (s->cc[CC_KMAX] - s->cc[CC_KMIN]);
    uint64_t u = mix64(mix64(((uint64_t)t << 32) | p->key) ^ ((uint64_t)qin << 40) ^ s->ecmp_seed) &
                 0xFFFFu;
    return u < prob;
}

/* Reaction point.  A rate increase event (the rate timer expired or B more
 * packets went out): fast recovery while both event counts are below F,
 * hyper increase once both exceed it, additive increase otherwise; the
 * current rate then moves halfway to the target, rounded up so that it
 * reaches the target. */
static void cc_increase(sim *s, lane *L)
{
    uint32_t mx = L->tc > L->bc ? L->tc : L->bc, mn = L->tc < L->bc ? L->tc : L->bc;
    uint32_t F = s->cc[CC_F];
    uint64_t rt = L->rt;
    if (mx < F) {
        /* fast recovery: the target stays */
    } else if (mn > F) {
        rt += (uint64_t)(mn - F) * s->cc[CC_RHAI];
    } else {
        rt += s->cc[CC_RAI];
    }
    L->rt = rt > CC_LINE ? CC_LINE : (uint32_t)rt;
    L->rc = (L->rt + L->rc + 1) / 2;
}

/* The timer events up to tick t, in time order (alpha first on a tie):
 * every K ticks without a notification alpha decays by the factor 1 - g;
 * every T ticks the rate timer fires a rate increase event.  Once alpha no
 * longer moves and both rates are at line rate, later events change
 * nothing but the timers' phase, so they are counted in one step. */
static void cc_catch_up(sim *s, lane *L, uint32_t t)
{
    const uint32_t K = s->cc[CC_K], T = s->cc[CC_T], gs = s->cc[CC_GSHIFT];
    for (;;) {
        if ((L->alpha >> gs) == 0 && L->rc == CC_LINE && L->rt == CC_LINE) {
            if (t >= L->abase) L->abase += (t - L->abase) / K * K;
            if (t >= L->rbase) {
                uint32_t n = (t - L->rbase) / T;
                L->rbase += n * T;
                L->tc = L->tc + n > 0xFFFFu ? 0xFFFFu : L->tc + n;
            }
            return;
        }
        uint64_t ta = (uint64_t)L->abase + K, tr = (uint64_t)L->rbase + T;
        if (ta > t && tr > t) return;
        if (ta <= tr) {
            L->alpha -= L->alpha >> gs;
            L->abase = (uint32_t)ta;
        } else {
            L->rbase = (uint32_t)tr;
            if (L->tc < 0xFFFFu) L->tc++;
            cc_increase(s, L);
        }
    }
}

/* A congestion notification reaching the lane at tick t: the target rate
 * becomes the current rate, the current rate drops by the factor
 * 1 - alpha/2 (not below the minimum rate), alpha moves to
 * (1 - g) alpha + g, and both timers and the byte counter restart. */
static void cc_cut(sim *s, lane *L, uint32_t r, uint32_t t)
{
    cc_catch_up(s, L, t);
    const uint32_t gs = s->cc[CC_GSHIFT];
    L->rt = L->rc;
    uint32_t dec = (uint32_t)(((uint64_t)L->rc * L->alpha) >> 21);
    L->rc = L->rc - dec < s->cc[CC_RMIN] ? s->cc[CC_RMIN] : L->rc - dec;
    L->alpha = L->alpha - (L->alpha >> gs) + (CC_LINE >> gs);
    if (L->alpha > CC_LINE) L->alpha = CC_LINE;
    L->abase = L->rbase = t;
    L->tc = L->bc = L->sent = 0;
    ev(s, EV_CUT, r, L->rc);
}

/* The lane sent a packet at tick t over an uplink of serialisation sigma:
 * the byte counter may fire a rate increase; the next packet may leave
 * once a packet's time at the current rate has passed. */
static void cc_sent(sim *s, lane *L, uint32_t sigma, uint32_t t)
{
    cc_catch_up(s, L, t);
    if (++L->sent >= s->cc[CC_B]) {
        L->sent = 0;
        if (L->bc < 0xFFFFu) L->bc++;
        cc_increase(s, L);
    }
    L->next_tx = t + (uint32_t)((((uint64_t)sigma << 20) + L->rc - 1) / L->rc);
}

/* Egress qe (egress i of P at its switch) sends packet p, taken from
 * ingress queue qin at tick t, to its downstream queue d: ready after the
 * link's serialisation and delay, one (delta + 1) more on the path's
 * acknowledgement delay; the egress is busy for sigma and its round-robin
 * pointer moves past the ingress it served. */
static void send_on(sim *s, uint32_t qe, uint32_t d, pkt p, uint32_t qin, uint32_t i, uint32_t P,
                    uint32_t t)
{
    if (s->cc[CC_ON] && !p.ecn && !p.cnp) p.ecn = ecn_mark(s, qin, &p, t);
    p.ready = t + s->port_sigma[qe] + s->port_delta[qe];
    p.hopsum += s->port_delta[qe] + 1;
    push(s, d, &p, t, s->port_sigma[qe]);
    ev(s, EV_HOP, qe, qin);
    s->eg_busy[qe] = t + s->port_sigma[qe];
    s->eg_rr[qe] = (i + 1) % P;
    s->pkt_hops++;
    s->changed = 1;
}

/* Switch forwarding with virtual output queues (the VOQ variant of the
 * pull-based forwarding, Multiverse section 4.2): an ingress buffer of cap
 * slots holds one FIFO per egress.  Plan: for each ingress, the oldest ready
 * packet for each egress (a buffer's packets are ready in arrival order, so
 * the scan stops at the first packet that is not).  Pull: the egresses in
 * index order; a free egress with credit downstream scans the ingress ports
 * round-robin from its pointer and takes the first one holding a ready
 * packet for it that no lower egress took a packet from in this tick (an
 * ingress sends at most one packet a tick).  A packet that leaves from the
 * middle of the buffer frees its slot when the buffer's head passes it, so
 * credit counts the span from the head to the tail as in the FIFO switch. */
static void voq_take(sim *s, uint32_t f, uint32_t x, uint32_t t)
{
    s->taken[f] |= 1ull << (x % s->cap);
    while (s->head[f] != s->tail[f] && ((s->taken[f] >> (s->head[f] % s->cap)) & 1ull)) {
        s->taken[f] &= ~(1ull << (s->head[f] % s->cap));
        pop(s, f, t);
    }
}

static void forward_voq(sim *s, uint32_t w, uint32_t t)
{
    uint32_t P = s->sw_nports[w], base = s->sw_base[w];
    uint32_t first[64][64];               /* [ingress][egress]: counter of its oldest ready packet */
    uint32_t wanted[64];
    memset(wanted, 0, sizeof(uint32_t) * P);
    for (uint32_t p = 0; p < P; p++) {
        uint32_t f = base + p;
        for (uint32_t e = 0; e < P; e++) first[p][e] = UNSET;
        for (uint32_t x = s->head[f]; x != s->tail0[f]; x++) {
            if ((s->taken[f] >> (x % s->cap)) & 1ull) continue;
            pkt *h = slot(s, f, x);
            if (h->ready > t) break;
            int32_t e = route_port(s, w, h);
            if (e < 0) { fail(s, ST_ERROR); continue; }     /* that packet stays */
            if (first[p][e] == UNSET) { first[p][e] = x; wanted[e]++; }
        }
    }
    uint64_t used = 0;                    /* ingresses a packet left this tick */
    for (uint32_t e = 0; e != P; e++) {   /* egresses in index order */
        uint32_t qe = base + e;
        if (!wanted[e] || t < s->eg_busy[qe]) continue;       /* nothing for it, or busy */
        uint32_t d = downstream(s, qe);
        if (!has_credit(s, d, t)) continue;
        for (uint32_t k = 0; k < P; k++) {
            uint32_t i = s->eg_rr[qe] + k;         /* round robin from the pointer */
            if (i >= P) i -= P;
            if (((used >> i) & 1ull) || first[i][e] == UNSET) continue;
            pkt p = *slot(s, base + i, first[i][e]);
            voq_take(s, base + i, first[i][e], t);
            s->sw_queued[w]--;
            send_on(s, qe, d, p, base + i, i, P, t);
            used |= 1ull << i;
            break;
        }
    }
}

/* Switch forwarding (Multiverse section 4.2, pull-based): plan = for each
 * ingress port, the egress its ready head packet needs; pull = each free
 * egress with credit downstream scans the ingress ports round-robin from its
 * pointer and takes the first head planned for it. */
static void forward(sim *s, uint32_t w, uint32_t t)
{
    if (s->sw_queued[w] == 0) return;     /* nothing queued: nothing to plan */
    if (s->voq) { forward_voq(s, w, t); return; }
    uint32_t P = s->sw_nports[w], base = s->sw_base[w];
    int32_t tgt[256];
    uint32_t wanted[256];                 /* how many heads want each egress */
    memset(wanted, 0, sizeof(uint32_t) * P);
    for (uint32_t p = 0; p < P; p++) {
        pkt *h = ready_head(s, base + p, t);
        tgt[p] = -1;
        if (h) {
            tgt[p] = route_port(s, w, h);
            if (tgt[p] < 0) { fail(s, ST_ERROR); continue; }   /* that head stays */
            wanted[tgt[p]]++;
        }
    }
    for (uint32_t e = 0; e < P; e++) {
        uint32_t qe = base + e;
        if (wanted[e] == 0 || s->eg_busy[qe] > t) continue;
        uint32_t d = downstream(s, qe);
        if (!has_credit(s, d, t)) continue;
        for (uint32_t k = 0; k < P; k++) {
            uint32_t i = (s->eg_rr[qe] + k) % P;
            if (tgt[i] != (int32_t)e) continue;
            pkt p = *slot(s, base + i, s->head[base + i]);
            pop(s, base + i, t);
            s->sw_queued[w]--;
            send_on(s, qe, d, p, base + i, i, P, t);
            break;
        }
    }
}

/* NIC send (SendSys + NICSndSys): one packet per uplink serialisation time,
 * round-robin over the rank's send lanes.  A lane may send when the receive
 * counts its current message waits for are reached (NCCL's step order), and
 * when the receiving rank joined the collective before this tick. */
static void inject(sim *s, uint32_t r, uint32_t t)
{
    nic *n = &s->nics[r];
    int cnps = n->cq_head != n->cq_tail;
    if ((n->n_lanes == 0 && !cnps) || n->busy > t) return;
    uint32_t f = s->host_port[r];
    if (!has_credit(s, f, t)) return;
    if (cnps) {
        /* a waiting congestion notification goes first; it takes one
         * packet time and leaves the round-robin pointer where it is */
        uint32_t k = n->cq_head++ % NCNPQ;
        const uint32_t sg = s->host_sigma[r], dl = s->host_delta[r];
        pkt p;
        memset(&p, 0, sizeof p);
        p.ready = t + sg + dl;
        p.dst = n->cq_dst[k];
        p.hopsum = dl + 1;
        p.key = n->cq_key[k];
        p.lane = n->cq_lane[k];
        p.cnp = 1;
        p.n = n->cq_n[k];
        p.m = n->cq_m[k];
        push(s, f, &p, t, sg);
        n->busy = t + sg;
        s->pkt_hops++;
        s->changed = 1;
        return;
    }
    /* occupied slots in round-robin order from the pointer: those at or
     * after it, then those before it */
    for (int pass = 0; pass < 2; pass++) {
        uint64_t m = pass == 0 ? (n->used_mask & (~0ULL << n->rr)) : (n->used_mask & ((1ULL << n->rr) - 1));
        while (m) {
            uint32_t q = (uint32_t)__builtin_ctzll(m);
            m &= m - 1;
            lane *L = &n->lanes[q];
            if (L->draining) continue;                      /* all sent: waits for its acks */
            int ok = 1;
            for (uint32_t b = 0; b < 3; b++)
                if ((L->dep_mask >> b) & 1u)
                    if (n->port_count[s->port_base[L->node] + L->dep_base + b] < L->dep_need) ok = 0;
            if (!ok) continue;
            uint32_t c = coll_of(s, L->node);
            uint32_t dnode = mnode(s, c, L->dst_member);
            /* rendezvous: the destination's join reaches this rank one
             * link latency (1 + smallest delta) after it happened */
            if (s->start[dnode] == UNSET || s->start[dnode] + s->rdv_delay > t) continue;
            if (s->cc[CC_ON] == CC_DCQCN && L->next_tx > t) continue;   /* paced by its rate */
            if (s->cc[CC_ON] == CC_DCTCP && L->sentc - L->acked >= L->wnd >> 10)
                continue;                                   /* its window is full */
            pkt p;
            p.ready = t + s->host_sigma[r] + s->host_delta[r];
            p.dst = mrank(s, c, L->dst_member);
            p.hopsum = s->host_delta[r] + 1;
            p.sender = L->node;
            p.pslot = s->port_base[dnode] + L->dst_port;
            p.last = L->pkts_left == 1;
            p.key = L->key;
            p.lane = q;
            p.ecn = p.cnp = p.n = p.m = 0;
            push(s, f, &p, t, s->host_sigma[r]);
            if (s->cc[CC_ON] == CC_DCQCN) cc_sent(s, L, s->host_sigma[r], t);
            if (s->cc[CC_ON] == CC_DCTCP) L->sentc++;
            ev(s, EV_INJECT, r, p.key);
            n->busy = t + s->host_sigma[r];
            n->rr = (q + 1) % NLANE;
            s->pkts_injected++;
            s->pkt_hops++;
            s->changed = 1;
            if (--L->pkts_left == 0) {
                if (++L->m == L->nmsg) {
                    if (s->cc[CC_ON] == CC_DCTCP) L->draining = 1;
                    else { L->used = 0; n->n_lanes--; n->used_mask &= ~(1ULL << q); }
                } else {
                    L->pkts_left = lane_setup(s, L);
                }
            }
            return;
        }
    }
}

/* DCTCP (Alizadeh et al., SIGCOMM 2010, an outside source: the Multiverse
 * page only names it).  An acknowledgement of n packets, m of them marked,
 * reaching lane q of rank r at tick t.  Once the packets sent before the
 * last window update are all acknowledged the observation window closes:
 * alpha <- (1 - g) alpha + g F with F the marked fraction of its
 * acknowledgements, and the window shrinks by the factor 1 - alpha/2 (not
 * below one packet) if any was marked, else grows by one packet (up to
 * Wmax).  A draining lane frees its slot once every packet is
 * acknowledged. */
static void dctcp_ack(sim *s, uint32_t r, uint32_t q, uint32_t na, uint32_t ma, uint32_t t)
{
    nic *n = &s->nics[r];
    lane *L = &n->lanes[q];
    if (!L->used) return;
    const uint32_t gs = s->cc[CC_GSHIFT];
    ev(s, EV_ACK, r, na | (ma << 8) | (q << 16));
    L->acked += na;
    L->wa += na;
    L->wm += ma;
    if (L->acked >= L->wend) {
        uint32_t F = (uint32_t)(((uint64_t)L->wm << 20) / L->wa);
        L->alpha = L->alpha - (L->alpha >> gs) + (F >> gs);
        if (L->wm) {
            uint32_t dec = (uint32_t)(((uint64_t)L->wnd * L->alpha) >> 21);
            L->wnd = L->wnd - dec < 1024 ? 1024 : L->wnd - dec;
        } else {
            L->wnd += 1024;
            if (L->wnd > s->cc[CC_WMAX] << 10) L->wnd = s->cc[CC_WMAX] << 10;
        }
        L->wa = L->wm = 0;
        L->wend = L->sentc;
        ev(s, EV_WINDOW, r, L->wnd);
    }
    if (L->draining && L->acked == L->sentc) {
        L->used = 0;
        n->n_lanes--;
        n->used_mask &= ~(1ULL << q);
    }
    (void)t;
}

/* NIC receive (NICRcvSys + ACKSys): the ready head of the NIC's downlink
 * queue.  The last packet of a message completes it: the receive count goes
 * up, the receiver's membership is one message closer to done, and the
 * sender's membership gets the message's acknowledgement, which reaches it
 * one propagation-plus-one-tick per hop after delivery. */
static void receive(sim *s, uint32_t r, uint32_t t)
{
    uint32_t f = q_of_host(s, r);
    pkt *h = ready_head(s, f, t);
    if (!h) return;
    pkt p = *h;
    if (p.dst != r) s->violations++;
    pop(s, f, t);
    s->changed = 1;
    nic *n = &s->nics[r];
    if (p.cnp && s->cc[CC_ON] == CC_DCTCP) {
        dctcp_ack(s, r, p.lane, p.n, p.m, t);
        return;
    }
    if (p.cnp) {
        /* reaction point: the notification reaches the lane it names; one
         * meant for an earlier flow of that slot is dropped */
        lane *L = &n->lanes[p.lane];
        if (L->used && L->key == p.key) cc_cut(s, L, r, t);
        return;
    }
    s->pkts_delivered++;
    ev(s, EV_DELIVER, r, p.sender);
    if (s->cc[CC_ON] == CC_DCTCP) {
        /* every data packet is acknowledged: the newest acknowledgement
         * still waiting for the same sender lane takes it over (up to 255
         * packets), else a new one joins the ring */
        uint32_t sr = s->node_rank[p.sender];
        for (uint32_t i = n->cq_tail; i != n->cq_head;) {
            uint32_t k = --i % NCNPQ;
            if (n->cq_dst[k] != sr || n->cq_lane[k] != p.lane) continue;
            if (n->cq_n[k] < 255) {
                n->cq_n[k]++;
                n->cq_m[k] += p.ecn;
                goto acked;
            }
            break;
        }
        if (n->cq_tail - n->cq_head >= NCNPQ) {
            fail(s, ST_OVERFLOW);                     /* the acknowledgement ring is full */
        } else {
            uint32_t k = n->cq_tail++ % NCNPQ;
            n->cq_dst[k] = sr;
            n->cq_lane[k] = p.lane;
            n->cq_key[k] = p.key;
            n->cq_n[k] = 1;
            n->cq_m[k] = p.ecn;
        }
    acked:;
    } else if (p.ecn) {
        /* notification point: at most one notification a flow per N ticks
         * (the flow's table entry remembers the last one); it waits in the
         * NIC's notification ring, which drops it when full */
        uint32_t j = p.key % NPTAB;
        if (!(n->np_key[j] == p.key && n->np_at[j] != UNSET &&
              (uint64_t)t < (uint64_t)n->np_at[j] + s->cc[CC_N]) &&
            n->cq_tail - n->cq_head < 16) {
            n->np_key[j] = p.key;
            n->np_at[j] = t;
            uint32_t k = n->cq_tail++ % NCNPQ;
            n->cq_dst[k] = s->node_rank[p.sender];
            n->cq_lane[k] = p.lane;
            n->cq_key[k] = p.key;
            n->cq_n[k] = n->cq_m[k] = 0;
            ev(s, EV_CNP, r, p.key);
        }
    }
    if (!p.last) return;
    ev(s, EV_MESSAGE, r, p.sender);
    n->port_count[p.pslot]++;
    uint32_t own = n->port_node[p.pslot];
    s->outstanding[own]--;
    s->done_max[own] = umax32(s->done_max[own], t);
    s->outstanding[p.sender]--;
    s->done_max[p.sender] = umax32(s->done_max[p.sender], t + p.hopsum);
    s->msgs_delivered++;
    s->digest += mix64(mix64((uint64_t)p.sender | ((uint64_t)p.key << 32)) ^ (uint64_t)t);
    if (s->rec_count < s->rec_cap) {
        s->rec_sender[s->rec_count] = p.sender;
        s->rec_key[s->rec_count] = p.key;
        s->rec_tick[s->rec_count] = t;
    }
    s->rec_count++;
}

/* ------------------------------------------------------------------------ */
/* GPU memory check (Multiverse section 3.1, "GPU memory simulator").  The
 * page gives no formula; this reads it as bf16 weights + gradients + fp32
 * Adam state (16 bytes per parameter) split over TP x PP, plus the
 * activations of min(m, PP) in-flight micro-batches of one pipeline stage
 * using the per-layer activation size s*b*h*(34 + 5*a*s/h) of Korthikanti et
 * al. 2022 (an outside source, named as such), split over TP. */
static int memory_fits(const uint64_t *mem, uint64_t cap)
{
    if (mem[9] == 0) return 1;
    uint64_t params = mem[0], tp = mem[1], pp = mem[2], layers = mem[3], m = mem[4];
    uint64_t sq = mem[5], b = mem[6], h = mem[7], a = mem[8];
    uint64_t weights = 16 * params / (tp * pp);
    uint64_t per_layer = sq * b * (34 * h + 5 * a * sq);
    uint64_t acts = layers * umin(m, pp) * per_layer / tp;
    return weights + acts <= cap;
}

/* ------------------------------------------------------------------------ */
static uint32_t next_event(sim *s, uint32_t t)
{
    uint32_t best = UNSET;
    for (uint32_t r = 0; r < s->R; r++) {
        nic *n = &s->nics[r];
        for (int k = 0; k < n->n_pend; k++)
            if (n->pend_start[k] > t && n->pend_start[k] < best) best = n->pend_start[k];
        if (n->busy > t && n->busy < best) best = n->busy;
    }
    for (uint32_t f = 0; f < s->nf; f++) {
        if (s->head[f] == s->tail[f]) continue;
        uint32_t rd = slot(s, f, s->head[f])->ready;
        if (rd > t && rd < best) best = rd;
    }
    for (uint32_t q = 0; q < s->Q; q++)
        if (s->eg_busy[q] > t && s->eg_busy[q] < best) best = s->eg_busy[q];
    /* credit still travelling back to a sender */
    for (uint32_t f = 0; f < s->nf; f++) {
        uint32_t h = s->head[f];
        for (uint32_t back = 0; back < h && back < 64; back++) {
            uint32_t at = s->poplog[(size_t)f * 64 + (h - 1 - back) % 64] + s->credit_delay[f];
            if (at <= t) break;
            if (at < best) best = at;
        }
    }
    /* a paced lane's next packet */
    if (s->cc[CC_ON] == CC_DCQCN)
        for (uint32_t r = 0; r < s->R; r++)
            for (int q = 0; q < NLANE; q++) {
                lane *L = &s->nics[r].lanes[q];
                if (L->used && L->next_tx > t && L->next_tx < best) best = L->next_tx;
            }
    /* a destination's join still on its way to a sending rank */
    for (uint32_t r = 0; r < s->R; r++) {
        nic *n = &s->nics[r];
        for (int q = 0; q < NLANE; q++) {
            if (!n->lanes[q].used) continue;
            uint32_t c = coll_of(s, n->lanes[q].node);
            uint32_t st = s->start[mnode(s, c, n->lanes[q].dst_member)];
            if (st != UNSET && st + s->rdv_delay > t && st + s->rdv_delay < best)
                best = st + s->rdv_delay;
        }
    }
    return best;
}

/* Tick 0: the DAG's roots are scheduled to start. */
static void sim_begin(sim *s)
{
    s->cur_rank = -1;
    for (uint32_t r = 0; r < s->R; r++)
        for (uint32_t u = s->rank_base[r]; u < s->rank_base[r + 1]; u++)
            if (s->node_npred[u] == 0) pend_add(s, r, u, 0);
    s->t_next = 0;
}

/* Step from s->t_next until the experiment stops or its clock reaches
 * `limit` (exclusive); a later call with a larger limit carries on exactly
 * as one longer call would. */
static void sim_advance(sim *s, uint32_t limit)
{
    uint32_t t = s->t_next;
    if (limit > TICK_LIMIT) limit = TICK_LIMIT;
    s->cur_rank = -1;
    while (s->status == ST_RUNNING) {
        if (s->nodes_left == 0) { s->status = ST_DONE; break; }
        if (t >= limit) break;
        s->now = t;
        memcpy(s->tail0, s->tail, sizeof(uint32_t) * s->nf);
        s->changed = 0;
        for (uint32_t r = 0; r < s->R; r++) {
            s->cur_rank = (int)r;
            dag_step(s, r, t);
        }
        s->cur_rank = -1;
        for (uint32_t w = 0; w < s->S; w++) forward(s, w, t);
        for (uint32_t r = 0; r < s->R; r++)
            if (!s->nics[r].tick_fail) inject(s, r, t);
        for (uint32_t r = 0; r < s->R; r++)
            if (!s->nics[r].tick_fail) receive(s, r, t);
        s->active++;
        if (s->status != ST_RUNNING) break;
        if (s->nodes_left == 0) { s->status = ST_DONE; t++; break; }
        if (s->changed) { t++; continue; }
        uint32_t nx = next_event(s, t);
        if (nx == UNSET) { s->status = ST_DEADLOCK; t++; break; }
        t = s->no_skip ? t + 1 : nx;
    }
    s->t_next = t;
}

/* ------------------------------------------------------------------------ */
static uint32_t *prefix(const uint32_t *cnt, uint32_t n)
{
    uint32_t *p = malloc(sizeof(uint32_t) * (n + 1));
    p[0] = 0;
    for (uint32_t i = 0; i < n; i++) p[i + 1] = p[i] + cnt[i];
    return p;
}

typedef struct offs {
    uint32_t *host, *sw, *port, *rank, *node, *edge, *coll, *memb, *a2a, *a2a_in;
} offs;

/* The inputs this simulator takes, checked before any run (-2 when a batch
 * breaks one): the limits the library's header documents, so that both
 * sides refuse the same batches.  Switches have 1..64 ports; a link's
 * serialisation time is 1..65535 ticks and its delay + 1 at most 64 ticks
 * (the pop log keeps 64 entries); hosts number 1..65535; a collective has
 * 1..65535 members and fewer than 2^40 bytes; every DAG edge joins nodes of
 * one rank and the predecessor counts match the edges; every membership
 * names a node of its own kind and rank; an experiment has 1..1024
 * channels, 2..1024 queue slots (at most 64 with virtual output queues) and
 * a chunk size whenever a network collective other than the relay needs
 * one. */
static int validate(const orc_batch *b, const offs *o)
{
    if (b->version != 1 || b->n_topos == 0 || b->n_works == 0) return -2;
    for (uint32_t t = 0; t < b->n_topos; t++) {
        uint32_t nh = b->topo_nhosts[t], ns = b->topo_nsw[t], nq = b->topo_nports[t];
        const uint32_t *np = b->sw_nports + o->sw[t], *lev = b->sw_level + o->sw[t];
        const int32_t *peer = b->port_peer + o->port[t];
        const uint32_t *hp = b->host_port + o->host[t];
        if (nh == 0 || nh > 65535 || ns == 0) return -2;
        uint64_t q = 0;
        for (uint32_t w = 0; w < ns; w++) {
            if (np[w] == 0 || np[w] > 64 || lev[w] == 0 || lev[w] > 250) return -2;
            q += np[w];
        }
        if (q != nq) return -2;
        for (uint32_t p = 0; p < nq; p++) {
            uint32_t sg = b->port_sigma[o->port[t] + p], dl = b->port_delta[o->port[t] + p];
            if (sg == 0 || sg > 65535 || dl > 63) return -2;
            if (peer[p] >= 0) {
                if ((uint32_t)peer[p] >= nq || peer[peer[p]] != (int32_t)p) return -2;
            } else {
                uint32_t h = (uint32_t)(-(peer[p] + 1));
                if (h >= nh || hp[h] != p) return -2;
            }
        }
        for (uint32_t h = 0; h < nh; h++) {
            uint32_t sg = b->host_sigma[o->host[t] + h], dl = b->host_delta[o->host[t] + h];
            if (hp[h] >= nq || peer[hp[h]] != -(int32_t)(h + 1)) return -2;
            if (sg == 0 || sg > 65535 || dl > 63) return -2;
        }
    }
    for (uint32_t w = 0; w < b->n_works; w++) {
        uint32_t nr = b->work_nranks[w], nn = b->work_nnodes[w], nco = b->work_ncolls[w];
        if (nn >= (1u << 25) - 256) return -2;  /* a packet names its sender's node in 25 bits */
        const uint32_t *cnt = b->rank_nnodes + o->rank[w];
        const uint32_t *kind = b->node_kind + o->node[w], *arg = b->node_arg + o->node[w];
        const uint32_t *nsucc = b->node_nsucc + o->node[w], *succ = b->succ + o->edge[w];
        uint64_t tot = 0, edges = 0;
        for (uint32_t r = 0; r < nr; r++) tot += cnt[r];
        if (tot != nn) return -2;
        for (uint32_t u = 0; u < nn; u++) edges += nsucc[u];
        if (edges != b->work_nedges[w]) return -2;
        uint32_t *rank_of = malloc(sizeof(uint32_t) * (nn + 1));
        uint32_t *indeg = calloc(nn + 1, sizeof(uint32_t));
        uint32_t *seen = calloc(nn + 1, sizeof(uint32_t));
        int bad = 0;
        for (uint32_t r = 0, u = 0; r < nr; r++)
            for (uint32_t k = 0; k < cnt[r]; k++) rank_of[u++] = r;
        for (uint32_t u = 0, j = 0; u < nn && !bad; u++) {
            if (kind[u] > K_NET) bad = 1;
            else if (kind[u] != K_COMPUTE && arg[u] >= nco) bad = 1;
            if (b->node_dur_hi[o->node[w] + u] < b->node_dur_lo[o->node[w] + u]) bad = 1;
            for (uint32_t k = 0; k < nsucc[u] && !bad; k++, j++) {
                if (succ[j] >= nn || rank_of[succ[j]] != rank_of[u]) bad = 1;
                else indeg[succ[j]]++;
            }
        }
        for (uint32_t u = 0; u < nn && !bad; u++)
            if (indeg[u] != b->node_npred[o->node[w] + u]) bad = 1;
        uint32_t m = o->memb[w], ra = o->a2a[w], ca = o->a2a_in[w];
        for (uint32_t c = 0; c < nco && !bad; c++) {
            uint32_t g = o->coll[w] + c, N = b->coll_nmembers[g], k = b->coll_kind[g];
            int intra = b->coll_intra[g] != 0;
            if (N == 0 || N > 65535 || k > C_A2A || b->coll_bytes[g] >= (1ull << 40)) { bad = 1; break; }
            if (intra && (b->coll_alpha[g] == 0 || b->coll_beta_den[g] == 0 ||
                          b->coll_beta_num[g] > (1u << 20))) { bad = 1; break; }
            if (!intra && k == C_RELAY && b->coll_parts[g] == 0) { bad = 1; break; }
            if (!intra && k == C_P2P && N != 2) { bad = 1; break; }
            if (m + N > o->memb[w + 1]) { bad = 1; break; }
            for (uint32_t i = 0; i < N && !bad; i++, m++) {
                uint32_t rr = b->member_rank[m], u = b->member_node[m];
                if (rr >= nr || u >= nn || rank_of[u] != rr || seen[u]) { bad = 1; break; }
                if (kind[u] != (intra ? K_INTRA : K_NET) || arg[u] != c) { bad = 1; break; }
                seen[u] = 1;
                uint32_t na = b->member_a2a_n[m], ni = b->member_a2a_in_n[m];
                if (ra + na > o->a2a[w + 1] || ca + ni > o->a2a_in[w + 1]) { bad = 1; break; }
                for (uint32_t j = 0; j < na; j++, ra++)
                    if (b->a2a_dst[ra] >= N || b->a2a_dst[ra] == i ||
                        b->a2a_bytes[ra] >= (1ull << 40)) bad = 1;
                for (uint32_t j = 0; j < ni; j++, ca++)
                    if (b->a2a_in_src[ca] >= N) bad = 1;
            }
        }
        if (!bad && (m != o->memb[w + 1] || ra != o->a2a[w + 1] || ca != o->a2a_in[w + 1])) bad = 1;
        for (uint32_t u = 0; u < nn && !bad; u++)
            if (kind[u] != K_COMPUTE && !seen[u]) bad = 1;
        const uint64_t *mm = b->mem + (size_t)10 * w;
        if (mm[9] && (mm[1] == 0 || mm[2] == 0)) bad = 1;
        free(rank_of); free(indeg); free(seen);
        if (bad) return -2;
    }
    for (uint32_t e = 0; e < b->n_exps; e++) {
        uint32_t ti = b->exp_topo[e], wi = b->exp_work[e];
        if (ti >= b->n_topos || wi >= b->n_works) return -2;
        if (b->work_nranks[wi] > b->topo_nhosts[ti] || b->exp_algo[e] > A_TREE ||
            b->exp_nc[e] == 0 || b->exp_nc[e] > 1024 || b->exp_pkt[e] == 0 ||
            b->exp_cap[e] < 2 || b->exp_cap[e] > 1024 || b->exp_tick_ps[e] == 0 ||
            b->exp_voq[e] > 1 || (b->exp_voq[e] && b->exp_cap[e] > 64))
            return -2;
        if (b->exp_cc) {
            const uint32_t *c = b->exp_cc + (size_t)CC_FIELDS * e;
            if (c[CC_ON] > CC_DCTCP) return -2;
            if (c[CC_ON] == CC_DCTCP &&
                (b->exp_voq[e] || c[CC_KMIN] != c[CC_KMAX] || c[CC_GSHIFT] == 0 ||
                 c[CC_GSHIFT] > 16 || c[CC_W0] == 0 || c[CC_WMAX] < c[CC_W0] ||
                 c[CC_WMAX] > 65535))
                return -2;
            if (c[CC_ON] == CC_DCQCN && (b->exp_voq[e] || c[CC_KMIN] > c[CC_KMAX] || c[CC_PMAX] > 65536 ||
                             c[CC_GSHIFT] == 0 || c[CC_GSHIFT] > 16 || c[CC_N] == 0 ||
                             c[CC_K] == 0 || c[CC_T] == 0 || c[CC_B] == 0 ||
                             c[CC_F] > 65535 || c[CC_RAI] > CC_LINE || c[CC_RHAI] > CC_LINE ||
                             c[CC_RMIN] == 0 || c[CC_RMIN] > CC_LINE))
                return -2;
        }
        if (b->exp_chunk[e] == 0)
            for (uint32_t c = o->coll[wi]; c < o->coll[wi + 1]; c++)
                if (!b->coll_intra[c] && b->coll_kind[c] != C_RELAY) return -2;
    }
    return 0;
}

/* Tables and tick-0 state of experiment e (nothing simulated yet). */
static void sim_setup(sim *s, const orc_batch *b, const offs *o, uint32_t e)
{
    memset(s, 0, sizeof *s);
    s->b = b;
    s->e = e;
    uint32_t ti = b->exp_topo[e], wi = b->exp_work[e];
    s->H = b->topo_nhosts[ti];
    s->S = b->topo_nsw[ti];
    s->Q = b->topo_nports[ti];
    s->sw_nports = b->sw_nports + o->sw[ti];
    s->sw_level = b->sw_level + o->sw[ti];
    s->port_peer = b->port_peer + o->port[ti];
    s->port_sigma = b->port_sigma + o->port[ti];
    s->port_delta = b->port_delta + o->port[ti];
    s->host_port = b->host_port + o->host[ti];
    s->host_sigma = b->host_sigma + o->host[ti];
    s->host_delta = b->host_delta + o->host[ti];
    s->sw_base = prefix(s->sw_nports, s->S);
    s->port_sw = malloc(sizeof(uint32_t) * (s->Q + 1));
    for (uint32_t w = 0; w < s->S; w++)
        for (uint32_t q = s->sw_base[w]; q < s->sw_base[w + 1]; q++) s->port_sw[q] = w;
    build_routes(s);

    s->R = b->work_nranks[wi];
    s->NN = b->work_nnodes[wi];
    uint32_t nco = b->work_ncolls[wi], nme = b->work_nmembers[wi];
    s->node_kind = b->node_kind + o->node[wi];
    s->node_arg = b->node_arg + o->node[wi];
    s->node_npred = b->node_npred + o->node[wi];
    s->node_dur_lo = b->node_dur_lo + o->node[wi];
    s->node_dur_hi = b->node_dur_hi + o->node[wi];
    s->node_dur_key = b->node_dur_key + o->node[wi];
    s->succ = b->succ + o->edge[wi];
    s->coll_kind = b->coll_kind + o->coll[wi];
    s->coll_intra = b->coll_intra + o->coll[wi];
    s->coll_bytes = b->coll_bytes + o->coll[wi];
    s->coll_nmembers = b->coll_nmembers + o->coll[wi];
    s->coll_parts = b->coll_parts + o->coll[wi];
    s->coll_alpha = b->coll_alpha + o->coll[wi];
    s->coll_beta_num = b->coll_beta_num + o->coll[wi];
    s->coll_beta_den = b->coll_beta_den + o->coll[wi];
    s->member_rank = b->member_rank + o->memb[wi];
    s->member_node = b->member_node + o->memb[wi];
    s->a2a_dst = b->a2a_dst + o->a2a[wi];
    s->a2a_bytes = b->a2a_bytes + o->a2a[wi];
    s->a2a_in_src = b->a2a_in_src + o->a2a_in[wi];
    s->a2a_in_bytes = b->a2a_in_bytes + o->a2a_in[wi];
    s->mem = b->mem + (size_t)10 * wi;
    s->rank_base = prefix(b->rank_nnodes + o->rank[wi], s->R);
    s->succ_base = prefix(b->node_nsucc + o->node[wi], s->NN);
    s->member_base = prefix(s->coll_nmembers, nco);
    s->row_base = prefix(b->member_a2a_n + o->memb[wi], nme);
    s->col_base = prefix(b->member_a2a_in_n + o->memb[wi], nme);
    s->node_rank = malloc(sizeof(uint32_t) * (s->NN + 1));
    s->node_member = calloc(s->NN + 1, sizeof(uint32_t));
    for (uint32_t r = 0; r < s->R; r++)
        for (uint32_t u = s->rank_base[r]; u < s->rank_base[r + 1]; u++) s->node_rank[u] = r;
    for (uint32_t c = 0; c < nco; c++)
        for (uint32_t i = 0; i < s->coll_nmembers[c]; i++) s->node_member[mnode(s, c, i)] = i;

    s->algo = b->exp_algo[e];
    s->nc = b->exp_nc[e];
    s->chunk = b->exp_chunk[e];
    s->pkt = b->exp_pkt[e];
    s->cap = b->exp_cap[e];
    s->tick_ps = b->exp_tick_ps[e];
    s->dur_seed = b->exp_dur_seed[e];
    s->ecmp_seed = b->exp_ecmp_seed[e];
    s->gpu_mem = b->exp_gpu_mem[e];
    s->rec_cap = b->exp_rec_cap[e];

    s->nf = s->Q + s->H;
    s->head = calloc(s->nf, sizeof(uint32_t));
    s->tail = calloc(s->nf, sizeof(uint32_t));
    s->tail0 = calloc(s->nf, sizeof(uint32_t));
    s->poplog = calloc((size_t)s->nf * 64, sizeof(uint32_t));
    s->credit_delay = calloc(s->nf, sizeof(uint32_t));
    s->rdv_delay = UNSET;
    for (uint32_t q = 0; q < s->Q; q++) {            /* switch ingress q: fed by its peer */
        int32_t pe = s->port_peer[q];
        uint32_t dl = pe >= 0 ? s->port_delta[pe] : s->host_delta[-pe - 1];
        s->credit_delay[q] = dl + 1;
        if (dl + 1 < s->rdv_delay) s->rdv_delay = dl + 1;
    }
    for (uint32_t h = 0; h < s->H; h++) {            /* NIC receive queue: fed by its switch port */
        uint32_t dl = s->port_delta[s->host_port[h]];
        s->credit_delay[s->Q + h] = dl + 1;
        if (dl + 1 < s->rdv_delay) s->rdv_delay = dl + 1;
    }
    s->slots = calloc((size_t)s->nf * s->cap, sizeof(pkt));
    s->last_push = malloc(sizeof(uint32_t) * s->nf);
    for (uint32_t f = 0; f < s->nf; f++) s->last_push[f] = UNSET;
    s->eg_busy = calloc(s->Q + 1, sizeof(uint32_t));
    s->eg_rr = calloc(s->Q + 1, sizeof(uint32_t));
    s->voq = b->exp_voq[e] != 0;
    if (b->exp_cc) memcpy(s->cc, b->exp_cc + (size_t)CC_FIELDS * e, sizeof s->cc);
    s->taken = calloc(s->Q + 1, sizeof(uint64_t));
    s->sw_queued = calloc(s->S + 1, sizeof(uint32_t));
    s->nics = calloc(s->R + 1, sizeof(nic));
    for (uint32_t r = 0; r <= s->R; r++)
        for (int j = 0; j < NPTAB; j++) s->nics[r].np_at[j] = UNSET;
    s->npred_left = malloc(sizeof(uint32_t) * (s->NN + 1));
    s->cand = calloc(s->NN + 1, sizeof(uint32_t));
    s->start = malloc(sizeof(uint32_t) * (s->NN + 1));
    s->end = malloc(sizeof(uint32_t) * (s->NN + 1));
    s->port_base = calloc(s->NN + 1, sizeof(uint32_t));
    s->done_max = calloc(s->NN + 1, sizeof(uint32_t));
    s->outstanding = calloc(s->NN + 1, sizeof(int64_t));
    for (uint32_t u = 0; u < s->NN; u++) {
        s->npred_left[u] = s->node_npred[u];
        s->start[u] = UNSET;
        s->end[u] = UNSET;
    }
    s->nodes_left = s->NN;
    s->status = ST_RUNNING;
    if (!memory_fits(s->mem, s->gpu_mem)) s->status = ST_OOM;
    else sim_begin(s);
}

/* Free what a sim owns: its dynamic state, and its tables unless it is a
 * clone that shares them. */
static void sim_teardown(sim *s)
{
    if (!s->is_clone) {
        free(s->sw_base); free(s->port_sw); free(s->route); free(s->up_base); free(s->up_port);
        free(s->rank_base); free(s->succ_base); free(s->member_base); free(s->row_base);
        free(s->col_base); free(s->node_rank); free(s->node_member); free(s->credit_delay);
    }
    free(s->head); free(s->tail); free(s->tail0); free(s->slots);
    free(s->poplog); free(s->last_push);
    free(s->eg_busy); free(s->eg_rr); free(s->taken); free(s->sw_queued); free(s->nics); free(s->npred_left); free(s->cand);
    free(s->start); free(s->end); free(s->port_base); free(s->done_max); free(s->outstanding);
}

static int run_one(const orc_batch *b, const offs *o, uint32_t e, uint32_t limit,
                   orc_out *out, uint64_t node_off, uint64_t rec_off, uint64_t coll_off,
                   orc_event *trace,
                   uint64_t trace_cap, uint64_t *trace_n, uint32_t flags)
{
    sim S_, *s = &S_;
    sim_setup(s, b, o, e);
    uint32_t nco = b->work_ncolls[b->exp_work[e]];
    s->trace = trace;
    s->trace_cap = trace_cap;
    s->no_skip = (flags & ORC_NO_SKIP) != 0;
    s->rec_sender = out->rec_sender + rec_off;
    s->rec_key = out->rec_key + rec_off;
    s->rec_tick = out->rec_tick + rec_off;
    if (s->status == ST_RUNNING) sim_advance(s, limit);
    uint64_t active = s->active;
    uint32_t now = s->t_next;

    uint32_t endt = 0;
    int any = 0;
    for (uint32_t u = 0; u < s->NN; u++) {
        out->node_start[node_off + u] = s->start[u];
        out->node_end[node_off + u] = s->end[u];
        if (s->end[u] != UNSET) { endt = umax32(endt, s->end[u]); any = 1; }
    }
    out->status[e] = (uint32_t)s->status;
    out->end_tick[e] = any ? endt : UNSET;
    /* the clock: where a stopped-by-budget experiment resumes; for one that
     * stopped for good, one past its latest node end (0 if none ended) */
    out->now[e] = s->status == ST_RUNNING ? now : (any ? endt + 1 : 0);
    out->pkts_injected[e] = s->pkts_injected;
    out->pkt_hops[e] = s->pkt_hops;
    out->pkts_delivered[e] = s->pkts_delivered;
    out->msgs_delivered[e] = s->msgs_delivered;
    out->digest[e] = s->digest;
    out->ticks_active[e] = active;
    out->rec_count[e] = s->rec_count;
    out->violations[e] = s->violations;
    /* Per-collective time (Multiverse section 3.1: the network simulator
     * tells the system simulator when each flow completes; a collective is
     * done when its last member is): from its first member's start to its
     * last member's end. */
    if (out->coll_start && out->coll_end) {
        for (uint32_t c = 0; c < nco; c++) {
            uint32_t lo = UNSET, hi = 0;
            int all_ended = 1;
            for (uint32_t i = 0; i < s->coll_nmembers[c]; i++) {
                uint32_t u = mnode(s, c, i);
                if (s->start[u] < lo) lo = s->start[u];
                if (s->end[u] == UNSET) all_ended = 0;
                else if (s->end[u] > hi) hi = s->end[u];
            }
            out->coll_start[coll_off + c] = lo;
            out->coll_end[coll_off + c] = all_ended ? hi : UNSET;
        }
    }
    if (trace_n) *trace_n = s->trace_n;
    sim_teardown(s);
    return 0;
}

/* Simulate experiments [e0, e1) of the batch (all of them when e1 == 0),
 * each to completion or until its clock reaches `limit` ticks.  Per-node
 * results go to node_start/node_end at the experiment's offset in the
 * concatenation of all experiments' nodes; flow records at the experiment's
 * offset in the concatenation of rec_cap-sized blocks. */
int orc_run_ex(const orc_batch *b, uint32_t e0, uint32_t e1, uint32_t limit, orc_out *out,
               orc_event *trace, uint64_t trace_cap, uint64_t *trace_n, uint32_t flags)
{
    offs o;
    o.host = prefix(b->topo_nhosts, b->n_topos);
    o.sw = prefix(b->topo_nsw, b->n_topos);
    o.port = prefix(b->topo_nports, b->n_topos);
    uint32_t *rank = prefix(b->work_nranks, b->n_works);
    o.rank = rank;
    o.node = prefix(b->work_nnodes, b->n_works);
    o.edge = prefix(b->work_nedges, b->n_works);
    o.coll = prefix(b->work_ncolls, b->n_works);
    o.memb = prefix(b->work_nmembers, b->n_works);
    o.a2a = prefix(b->work_na2a, b->n_works);
    o.a2a_in = prefix(b->work_na2a_in, b->n_works);
    if (e1 == 0 || e1 > b->n_exps) e1 = b->n_exps;
    int bad = validate(b, &o);
    uint64_t node_off = 0, rec_off = 0, coll_off = 0;
    for (uint32_t e = 0; e < e1 && !bad; e++) {
        if (e >= e0)
            run_one(b, &o, e, limit, out, node_off, rec_off, coll_off, trace, trace_cap,
                    trace_n, flags);
        node_off += b->work_nnodes[b->exp_work[e]];
        rec_off += b->exp_rec_cap[e];
        coll_off += b->work_ncolls[b->exp_work[e]];
    }
    free(o.host); free(o.sw); free(o.port); free(rank); free(o.node); free(o.edge);
    free(o.coll); free(o.memb); free(o.a2a); free(o.a2a_in);
    return bad;
}

/* Without a trace and with idle ticks skipped.  orc_run_ex: with a trace,
 * give e1 = e0 + 1 (the events of one experiment; *trace_n gets how many
 * happened); flags ORC_NO_SKIP steps every tick one by one (the brute-force
 * check that skipping idle ticks changes no result). */
int orc_run(const orc_batch *b, uint32_t e0, uint32_t e1, uint32_t limit, orc_out *out)
{
    return orc_run_ex(b, e0, e1, limit, out, NULL, 0, NULL, 0);
}

/* exported for the tests that pin the hash against its published values */
uint64_t orc_mix64(uint64_t z) { return mix64(z); }

/* ------------------------------------------------------------------------ */
/* A paused run of one experiment, so that a window of ticks can be timed on
 * its own: create (tick 0), advance to a tick, copy the state, advance the
 * copy.  This is plumbing around the same simulation steps; it keeps no
 * per-message records and no trace.  The batch arrays must outlive it. */
typedef struct orc_handle {
    sim s;
} orc_handle;

void *orc_sim_new(const orc_batch *b, uint32_t e)
{
    if (e >= b->n_exps) return NULL;
    offs o;
    o.host = prefix(b->topo_nhosts, b->n_topos);
    o.sw = prefix(b->topo_nsw, b->n_topos);
    o.port = prefix(b->topo_nports, b->n_topos);
    o.rank = prefix(b->work_nranks, b->n_works);
    o.node = prefix(b->work_nnodes, b->n_works);
    o.edge = prefix(b->work_nedges, b->n_works);
    o.coll = prefix(b->work_ncolls, b->n_works);
    o.memb = prefix(b->work_nmembers, b->n_works);
    o.a2a = prefix(b->work_na2a, b->n_works);
    o.a2a_in = prefix(b->work_na2a_in, b->n_works);
    orc_handle *h = NULL;
    if (validate(b, &o) == 0) {
        h = calloc(1, sizeof *h);
        sim_setup(&h->s, b, &o, e);
        h->s.rec_cap = 0;
    }
    free(o.host); free(o.sw); free(o.port); free(o.rank); free(o.node); free(o.edge);
    free(o.coll); free(o.memb); free(o.a2a); free(o.a2a_in);
    return h;
}

/* Advance to `limit` (exclusive); returns the experiment's status. */
int orc_sim_advance(void *hp, uint32_t limit)
{
    orc_handle *h = hp;
    if (h->s.status == ST_RUNNING) sim_advance(&h->s, limit);
    return h->s.status;
}

/* status, clock (the next tick the run would simulate), packets injected,
 * packet-hops, packets delivered, messages delivered */
void orc_sim_counters(void *hp, uint64_t *out)
{
    sim *s = &((orc_handle *)hp)->s;
    out[0] = (uint64_t)s->status;
    out[1] = s->t_next;
    out[2] = s->pkts_injected;
    out[3] = s->pkt_hops;
    out[4] = s->pkts_delivered;
    out[5] = s->msgs_delivered;
}

static void *dup_bytes(const void *src, size_t n)
{
    void *d = malloc(n ? n : 1);
    if (n) memcpy(d, src, n);
    return d;
}

/* A copy of the dynamic state; the read-only tables are shared with the
 * original, which must outlive the copy. */
void *orc_sim_clone(void *hp)
{
    const sim *a = &((orc_handle *)hp)->s;
    orc_handle *h = calloc(1, sizeof *h);
    sim *s = &h->s;
    *s = *a;
    s->is_clone = 1;
    s->head = dup_bytes(a->head, sizeof(uint32_t) * a->nf);
    s->tail = dup_bytes(a->tail, sizeof(uint32_t) * a->nf);
    s->tail0 = dup_bytes(a->tail0, sizeof(uint32_t) * a->nf);
    s->poplog = dup_bytes(a->poplog, sizeof(uint32_t) * (size_t)a->nf * 64);
    s->slots = dup_bytes(a->slots, sizeof(pkt) * (size_t)a->nf * a->cap);
    s->last_push = dup_bytes(a->last_push, sizeof(uint32_t) * a->nf);
    s->eg_busy = dup_bytes(a->eg_busy, sizeof(uint32_t) * (a->Q + 1));
    s->eg_rr = dup_bytes(a->eg_rr, sizeof(uint32_t) * (a->Q + 1));
    s->taken = dup_bytes(a->taken, sizeof(uint64_t) * (a->Q + 1));
    s->sw_queued = dup_bytes(a->sw_queued, sizeof(uint32_t) * (a->S + 1));
    s->nics = dup_bytes(a->nics, sizeof(nic) * (a->R + 1));
    s->npred_left = dup_bytes(a->npred_left, sizeof(uint32_t) * (a->NN + 1));
    s->cand = dup_bytes(a->cand, sizeof(uint32_t) * (a->NN + 1));
    s->start = dup_bytes(a->start, sizeof(uint32_t) * (a->NN + 1));
    s->end = dup_bytes(a->end, sizeof(uint32_t) * (a->NN + 1));
    s->port_base = dup_bytes(a->port_base, sizeof(uint32_t) * (a->NN + 1));
    s->done_max = dup_bytes(a->done_max, sizeof(uint32_t) * (a->NN + 1));
    s->outstanding = dup_bytes(a->outstanding, sizeof(int64_t) * (a->NN + 1));
    return h;
}

void orc_sim_free(void *hp)
{
    if (!hp) return;
    sim_teardown(&((orc_handle *)hp)->s);
    free(hp);
}
