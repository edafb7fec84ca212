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
constexpr u32 kPopLog = 64;    // pops remembered per queue (credit delay <= 64)

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
};

struct WorkRec {
    u32 nr, nn, ncoll, nmemb;
    u32 rank_off, node_off, edge_off, coll_off, memb_off, a2a_off, a2a_in_off, pad;
};

struct ExpRec {
    u32 topo, work, algo, nc, pkt, cap, tick_ps, rec_cap;
    u64 chunk, dur_seed, ecmp_seed, gpu_mem;
    u64 q_off;      // first queue (switch ingress queues, then NIC receive queues)
    u64 slot_off;   // first packet slot (queue-major, cap slots per queue)
    u64 eg_off;     // first egress record (one per switch port)
    u64 rk_off;     // first rank
    u64 nd_off;     // first node
    u64 rec_off;    // first message record
    u32 nq, nsw, nr, nn;
    u32 item_off;   // first work item (switches, then groups of 32 ranks)
    u32 n_items, pad0, pad1;
};

// One send lane: a stream of messages one rank sends for one channel of one
// collective membership (a queue pair in RDMA terms).
struct Lane {
    u32 node, member, chan, kind;
    u32 m, nmsg, pkts_left, dst_member;
    u32 dst_port, dep_base, dep_mask, dep_need;
    u32 key, a2a_e, a2a_start, pad;
};

struct RankCtl {
    u32 busy, rr, npend, nact;
    u64 lane_mask;
    u64 port_mask[2];
    u64 pad;
};

struct ExpCtl {
    u32 status, now, limit, nodes_left;
    u32 clk[3];              // tick processed at step k (slot k % 3)
    u32 nxt[3];              // min over pending wake ticks reported at step k
    u32 rec_count;
    u32 stop_step;           // first step in which it finished or failed
    u32 end_max1;            // 1 + latest node end tick (0: none yet)
    u32 pad;
    u64 pkts_injected, pkt_hops, pkts_delivered, msgs_delivered, digest;
};

struct Glob {
    u32 bar_count, bar_gen, error, run_cnt[3];
    u64 steps;
    u32 err_step, err_block;
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
    // dynamic state
    u64 *q_push, *q_pop;     // per queue: (tick << 32) | counter of the last push / pop
    u32 *poplog;             // per queue: tick of each of the last 64 pops (by head % 64)
    uint4 *slots;            // packet descriptors
    uint2 *eg;               // per switch port: (busy_until, round-robin pointer)
    RankCtl *rk;
    uint2 *pend;             // per rank: kNPend (node, start tick)
    u32 *act;                // per rank: kNAct running nodes, ascending
    Lane *lanes;             // per rank: kNLane
    uint2 *ports;            // per rank: kNPort (messages received, owner node)
    u32 *nd_pred, *nd_cand, *nd_start, *nd_end, *nd_pbase, *nd_done;
    i32 *nd_out;
    ExpCtl *ctl;
    u32 *rec_sender, *rec_key, *rec_tick;
    const u32 *item_exp, *item_loc;
    u32 *wake;               // per work item: earliest tick it may have work
    const u32 *node_rank;    // per node: its rank (workload-local)
    u32 n_items, n_exps, n_topos, pad;
    Glob *glob;
    // run options
    u64 barrier_timeout_ns;
    i32 fault_block, fault_step;
};

// Packet descriptor (16 bytes):
//   x ready tick | y dst host (16 b) + accumulated (delta+1) over hops (16 b)
//   z sender node | w connection key (24 b) + last flag (1 b) + receive slot (7 b)
__host__ __device__ inline u32 pk_dst(uint4 p) { return p.y & 0xFFFFu; }
__host__ __device__ inline u32 pk_hops(uint4 p) { return p.y >> 16; }
__host__ __device__ inline u32 pk_key(uint4 p) { return p.w & 0xFFFFFFu; }
__host__ __device__ inline u32 pk_last(uint4 p) { return (p.w >> 24) & 1u; }
__host__ __device__ inline u32 pk_slot(uint4 p) { return p.w >> 25; }

// launch wrappers (mv_kernel.cu)
cudaError_t launch_routes(const Params &p, u64 n_pairs_max, u32 level, cudaStream_t st);
cudaError_t launch_up_lists(const Params &p, u32 n_sw_total, cudaStream_t st);
cudaError_t launch_init(const Params &p, u32 max_nodes, u32 max_queues, u32 max_ranks,
                        cudaStream_t st);
cudaError_t launch_run_reset(const Params &p, u32 max_ticks, cudaStream_t st);
cudaError_t launch_megakernel(const Params &p, u32 blocks, cudaStream_t st);
cudaError_t megakernel_occupancy(int *blocks_per_sm, int *n_sm);

}  // namespace mv
