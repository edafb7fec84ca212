// mv_device.cuh -- device-side layout of the SPME packet simulator.
//
// Every experiment of a batch owns its own slice of each state array
// (structure of arrays, one slot per experiment and entity, Multiverse
// section 3.3); static topology and workload tables are shared by all the
// experiments that use them.  This header is internal to the library.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mv {

typedef uint32_t u32;
typedef uint64_t u64;
typedef int32_t i32;
typedef uint8_t u8;

constexpr u32 kUnset = 0xFFFFFFFFu;
constexpr u32 kNLane = 64;    // send lanes per rank (bit mask in RankCtl)
constexpr u32 kNPort = 128;   // receive counters per rank
constexpr u32 kNPend = 64;    // nodes scheduled to start, per rank
constexpr u32 kNAct = 16;     // running collective memberships, per rank
constexpr u32 kMaxPorts = 64; // ports per switch (one warp, two ports a lane)
constexpr u32 kTickLimit = 0xFFF00000u;
constexpr u32 kPopLog = 64;   // credit delay (delta + 1) of a link is at most this
constexpr u32 kMaxWarps = 32; // warps of the block that steps one experiment (build 4; 16 for
                              // build 3; 8 otherwise)

enum : u32 { NODE_COMPUTE = 0, NODE_INTRA = 1, NODE_NET = 2 };
enum : u32 { COLL_AR = 0, COLL_RS = 1, COLL_AG = 2, COLL_RELAY = 3, COLL_P2P = 4, COLL_A2A = 5 };
enum : u32 { ALGO_RING = 0, ALGO_TREE = 1 };
enum : u32 { EXP_DONE = 0, EXP_RUNNING = 1, EXP_OOM = 2, EXP_DEADLOCK = 3, EXP_OVERFLOW = 4,
             EXP_ERROR = 5 };

struct TopoRec {
    u32 nh, nsw, nq, maxlev;        // hosts, switches, switch ports, top level
    u32 host_off, sw_off, port_off;
    u32 rdv;                        // 1 + smallest link delta: how late a join reaches peers
    u64 route_off;                  // route table: nsw * nh bytes
    u32 plog;                       // pop-log entries per queue: power of two >= largest delta + 1
    u32 pad;
};

struct WorkRec {
    u32 nr, nn, ncoll, nmemb;
    u32 rank_off, node_off, edge_off, coll_off, memb_off, a2a_off, a2a_in_off, pad;
};

// One experiment: parameters, and where its slice of each dynamic array
// starts (element offsets).  Per-rank tables have per-experiment strides
// (lane_cap, port_cap, pend_cap, act_cap): the smaller of the fixed limit
// and what the experiment's DAG can ever need, so small experiments fit in
// shared memory while the limits (and the overflow status) are unchanged.
struct ExpRec {
    u32 topo, work, algo, nc, pkt, cap, tick_ps, rec_cap;
    u64 chunk, dur_seed, ecmp_seed, gpu_mem;
    u64 q_off, slot_off, plog_off, eg_off, rk_off, pend_off, act_off, lane_off, portc_off,
        nd_off, rec_off, coll_res_off, taken_off;
    u32 nq, nsw, nr, nn;            // queues (switch ingress, then NIC receive), switches, ranks, nodes
    u32 item_off, n_items;          // work items: switches, then groups of 32 ranks
    u32 lane_cap, port_cap, pend_cap, act_cap;
    u32 stage_bytes;                // bytes of the whole dynamic state as one shared-memory image
    u32 voq;                        // 1: switches keep virtual output queues
    u32 plog;                       // pop-log entries per queue: the fabric's, or 64 with VOQs
    u32 cc;                         // DCQCN: 0 = none, else 1 + its parameter record's index
    u64 lcc_off, rcc_off;           // with DCQCN: its lanes' rate records, its ranks' records
};

// Congestion control of an experiment, in the simulator's units.  mode 1,
// DCQCN: marking thresholds (packets) and top probability (2^-16), gain
// shift, notification gap N, alpha timer K and rate timer T (ticks), byte
// counter B (packets), fast-recovery count F, additive / hyper / minimum
// rate (2^-20 of the line rate).  mode 2, DCTCP: the marking threshold
// (kmin = kmax), gain shift, initial and largest window (packets).
constexpr u32 kDcqcn = 1, kDctcp = 2;
struct CcRec {
    u32 kmin, kmax, pmax, gshift, n, k, t, b, f, rai, rhai, rmin, w0, wmax, mode, pad;
};
constexpr u32 kLine = 1u << 20;      // the line rate (and alpha = 1) in DCQCN units

// A send lane's congestion-control state (32 bytes, beside its hot and cold
// records).  DCQCN reaction point: a = current rate, target rate, alpha,
// earliest tick of its next packet; b = alpha timer's and rate timer's last
// expiry, rate-timer events | byte-counter events << 16, packets since the
// last byte event.  DCTCP sender: a = window (2^-10 packets), alpha,
// packets sent, packets acknowledged; b = acknowledged count that closes
// the observation window, its acknowledgements, its marks, draining (all
// sent, waiting for acknowledgements).
struct LaneCC {
    uint4 a, b;
};

// A rank's congestion-control state at the receiving side: DCQCN's last
// notification per flow (direct-mapped by key mod 64: key | 1 << 31, tick),
// and the ring of control packets waiting to be sent (sender rank | its
// lane << 16 | packets acknowledged << 22, key | of them marked << 24):
// DCQCN notifications (at most kCnpRing of them) or DCTCP acknowledgements.
constexpr u32 kNpTab = 64, kCnpRing = 16, kCtlRing = 64;
struct RankCC {
    uint2 np[kNpTab];
    uint2 cq[kCtlRing];
    u32 head, tail, pad0, pad1;
};

// One send lane: a stream of messages one rank sends for one channel of one
// collective membership (a queue pair in RDMA terms), kept as two 32-byte
// records in two arrays.  The hot record holds everything a packet needs
// and is the only one read and written per packet (one 32-byte sector); the
// cold record holds what a new message needs (the collective, its member
// count, kind and first member entry, the message count and the all-to-all
// position).  Field packing (mv_kernel.cu, load_lane_hot / load_lane_cold):
//   hot  a: node, connection key | dep_mask << 24 | ok_dst << 27, packets left,
//           destination rank | destination slot << 16 | dst_port << 24
//        b: dep_need, dep_base | receive-counter base << 8 | chan << 16 | kind << 24,
//           destination node, message
//   cold a: collective, members | member << 16, first member entry, messages
//        b: destination member | coll kind << 16, a2a entry, a2a first chunk, 0
struct LaneHot {
    uint4 a, b;
};
struct LaneCold {
    uint4 a, b;
};

// Per-rank control word as stored (48 bytes).
struct RankCtl {
    u32 busy, rr, npend, nact;
    u64 lane_mask;
    u64 port_lo, port_hi;   // receive counters in use: bits 0..63, 64..127
    u32 flags;      // bit 0: every send lane waits for a receive count (no scan
                    // needed); bits 1..: running intra-server memberships
    u32 pfirst;     // start tick of the first pending node (kUnset: none)
};

// Per-experiment control, kept across runs (resume) and read by mv_results.
struct ExpCtl {
    u32 status, now, nodes_left, end_max1;   // end_max1 = 1 + latest node end (0: none yet)
    u32 rec_count, pad0, pad1, pad2;
    u64 pkts_injected, pkt_hops, pkts_delivered, msgs_delivered, digest;
};

struct Glob {
    u32 next;       // next slot of the processing order to hand out
    u32 error;      // set by the watchdog: blocks stop at their next tick boundary
    u32 err_exp, pad;
    u64 steps;      // most ticks one experiment processed in the last run
};

struct Params {
    // static tables
    const TopoRec *topo;
    const WorkRec *work;
    const ExpRec *exp;
    const u32 *sw_nports, *sw_level, *sw_pstart, *port_sw;
    const i32 *port_peer;
    const u32 *port_sigma, *port_delta, *host_port, *host_sigma, *host_delta;
    u8 *route, *up_n, *up_list;
    const u32 *rank_first, *rank_nnodes, *node_kind, *node_arg, *node_npred, *node_nsucc,
        *succ_start, *node_dur_lo, *node_dur_hi, *node_dur_key, *succ, *node_member;
    const u32 *coll_kind, *coll_intra, *coll_nmembers, *coll_parts, *coll_alpha,
        *coll_beta_num, *coll_beta_den, *coll_mstart;
    const u64 *coll_bytes;
    const u32 *member_rank, *member_node, *member_a2a_n, *memb_row, *a2a_dst,
        *member_a2a_in_n, *memb_col, *a2a_in_src;
    const u64 *a2a_bytes, *a2a_in_bytes, *mem;
    const u32 *node_rank;    // per node: its rank (workload-local)
    const uint2 *sw_rec;     // per switch: (first port, ports)
    const uint4 *port_rec;   // per switch port: (downstream queue, sigma, delta, owner of that
                             //   queue: peer switch, or 0x80000000 | host)
    const uint4 *host_rec;   // per host: (uplink queue, sigma, delta, switch of that queue)
    const u32 *order;        // experiments in the order blocks take them (largest first)
    // dynamic state
    u64 *q_push, *q_pop;     // per queue: (tick << 32) | counter of the last push / pop
    u64 *q_taken;            // with VOQs, per switch ingress queue: slots already forwarded
    u32 *poplog;             // per queue: tick of each of the last plog pops (by head % plog)
    uint4 *slots;            // packet descriptors
    uint2 *eg;               // per switch port: (busy_until, round-robin pointer)
    RankCtl *rk;
    u32 *rdirty;             // per rank: one of its running memberships has no message left
    uint2 *pend;             // per rank: pend_cap (node, start tick)
    u32 *act;                // per rank: act_cap running nodes, ascending
    LaneHot *lhot;           // per rank: lane_cap hot lane records
    LaneCold *lcold;         // per rank: lane_cap cold lane records
    uint2 *ports;            // per rank: port_cap (messages received, owner node)
    u32 *nd_pred, *nd_cand, *nd_start, *nd_end, *nd_pbase, *nd_done;
    i32 *nd_out;
    ExpCtl *ctl;
    u32 *rec_sender, *rec_key, *rec_tick;
    u32 *coll_start, *coll_end;  // per experiment and collective: first member start, last end
    const CcRec *ccrec;      // DCQCN parameter records (ExpRec::cc - 1)
    LaneCC *lcc;             // per lane of a DCQCN experiment: its reaction point
    RankCC *rcc;             // per rank of a DCQCN experiment: its notification point
    u32 *wake;               // per experiment: own wake tick of each item, then two poke words each
    u32 n_exps, n_topos;
    Glob *glob;
    // run options
    u64 watchdog_ns;         // 0 = none
    u32 max_ticks;           // tick budget of this run, per experiment clock
    u32 stage_limit;         // bytes of shared memory for an experiment's image
    u32 stage_mode;          // 0 = whole image when it fits, 1 = wake table only, 2 = none
    u32 pad;
};

// Packet descriptor (16 bytes):
//   x ready tick | y dst host (16 b) + accumulated (delta+1) over hops (16 b)
//   z sender node (25 b) + sender lane (6 b) + congestion mark (1 b)
//   w connection key (24 b) + last flag (1 b) + receive slot (7 b)
// A control packet (a DCQCN notification, a DCTCP acknowledgement) carries
// node kCtlNode + the packets it acknowledges (0 for a notification), the
// lane it is for, and in w the flow key and the marked packets it
// acknowledges (bits 24..31).
constexpr u32 kCtlNode = 0x1FFFF00u;
__host__ __device__ inline u32 pk_dst(uint4 p) { return p.y & 0xFFFFu; }
__host__ __device__ inline u32 pk_node(uint4 p) { return p.z & 0x1FFFFFFu; }
__host__ __device__ inline u32 pk_lane(uint4 p) { return (p.z >> 25) & 63u; }
__host__ __device__ inline u32 pk_ecn(uint4 p) { return p.z >> 31; }
__host__ __device__ inline u32 pk_hops(uint4 p) { return p.y >> 16; }
__host__ __device__ inline u32 pk_key(uint4 p) { return p.w & 0xFFFFFFu; }
__host__ __device__ inline u32 pk_last(uint4 p) { return (p.w >> 24) & 1u; }
__host__ __device__ inline u32 pk_slot(uint4 p) { return p.w >> 25; }

// Shared-memory image of one experiment: byte offsets of each array
// (16-byte aligned), in this order.  The wake table comes first, so an
// image cut after it holds the wake table alone.  The dynamic state
// (IM_WAKE .. IM_SLOTS) is copied in and back out; the topology records and
// routing tables after it are only copied in.
enum : int { IM_WAKE, IM_QPUSH, IM_QPOP, IM_EG, IM_RK, IM_RDIRTY, IM_PRED, IM_CAND, IM_START, IM_END,
             IM_PBASE, IM_DONE, IM_OUT, IM_ACT, IM_PEND, IM_PORTS, IM_POPLOG, IM_LHOT,
             IM_LCOLD, IM_TAKEN, IM_SLOTS, IM_NDYN, IM_SWREC = IM_NDYN, IM_PORTREC, IM_HOSTREC, IM_ROUTE, IM_UPN,
             IM_UPLIST, IM_N };

__host__ __device__ inline u64 im_round(u64 b) { return (b + 15) & ~15ull; }

__host__ __device__ inline void image_bytes(const ExpRec &X, const TopoRec &T, u64 *sz)
{
    const u32 plog = X.plog, n_eg = T.nq;
    sz[IM_WAKE] = 12ull * X.n_items;          // own wake + two poke words per item
    sz[IM_QPUSH] = 8ull * X.nq;
    sz[IM_QPOP] = 8ull * X.nq;
    sz[IM_EG] = 8ull * n_eg;
    sz[IM_RK] = sizeof(RankCtl) * (u64)X.nr;
    sz[IM_RDIRTY] = 4ull * X.nr;
    for (int k = IM_PRED; k <= IM_OUT; k++) sz[k] = 4ull * X.nn;
    sz[IM_ACT] = 4ull * X.nr * X.act_cap;
    sz[IM_PEND] = 8ull * X.nr * X.pend_cap;
    sz[IM_PORTS] = 8ull * X.nr * X.port_cap;
    sz[IM_POPLOG] = 4ull * X.nq * plog;
    sz[IM_LHOT] = sizeof(LaneHot) * (u64)X.nr * X.lane_cap;
    sz[IM_LCOLD] = sizeof(LaneCold) * (u64)X.nr * X.lane_cap;
    sz[IM_TAKEN] = X.voq ? 8ull * T.nq : 0;
    sz[IM_SLOTS] = 16ull * X.nq * X.cap;
    sz[IM_SWREC] = 8ull * T.nsw;
    sz[IM_PORTREC] = 16ull * T.nq;
    sz[IM_HOSTREC] = 16ull * T.nh;
    sz[IM_ROUTE] = (u64)T.nsw * T.nh;
    sz[IM_UPN] = T.nsw;
    sz[IM_UPLIST] = T.nq;
}

// offsets into the image; returns the total
__host__ __device__ inline u64 image_layout(const ExpRec &X, const TopoRec &T, u64 *off)
{
    u64 sz[IM_N];
    image_bytes(X, T, sz);
    u64 o = 0;
    for (int k = 0; k < IM_N; k++) {
        off[k] = o;
        o += im_round(sz[k]);
    }
    return o;
}

// launch wrappers (mv_kernel.cu)
cudaError_t launch_routes(const Params &p, u64 n_pairs_max, u32 level, cudaStream_t st);
cudaError_t launch_up_lists(const Params &p, u32 n_sw_total, cudaStream_t st);
cudaError_t launch_init(const Params &p, u32 max_nodes, u32 max_queues, u32 max_ranks,
                        cudaStream_t st);
cudaError_t launch_coll_times(const Params &p, u32 max_colls, cudaStream_t st);
// variant 1: latency (one block of <= 8 warps an SM, register view); 2: occupancy (two
// blocks of 8 warps an SM); 3: one block of 16 warps an SM (more shared memory a block);
// 4: one block of 32 warps an SM (64 registers a thread)
// cc: the build with the DCQCN code (needed when an experiment has DCQCN)
cudaError_t megakernel_prepare(u32 variant, bool cc, u32 warps, u32 smem_bytes,
                               int *blocks_per_sm, int *n_sm);
u32 megakernel_smem(u32 warps, u32 image_bytes);
u32 megakernel_scratch_bytes();   // per-warp forwarding scratch
cudaError_t launch_megakernel(u32 variant, bool cc, const Params &p, u32 blocks, u32 warps,
                              u32 smem_bytes, cudaStream_t st);

}  // namespace mv
