/*
 * mv.h -- C ABI of the GB300 single-process multi-experiment (SPME) packet
 * simulator of LLM-training collective traffic.
 *
 * Source of the operation: "Accelerating Design Space Exploration for LLM
 * Training Systems with Multi-experiment Parallel Simulation" (Multiverse,
 * NSDI'25).  Section 3.1 (architecture): the user describes the workload,
 * the collective-library parameters and the topology, lists the experiments,
 * and the simulator runs them all in one process on one GPU.  Section 3.2
 * fixes the per-step system order (Schedule, AnalyticalSys, SendSys,
 * NICSndSys, ForwardSys, TransmitSys, NICRcvSys, ACKSys), section 3.3 the
 * per-experiment columnar state, section 4.2 the pull-based forwarding and
 * section 4.3 the single megakernel launched once per batch.  The collective
 * parameters <algorithm, NC, C> are AutoCCL's (section 2.3); the pipelined
 * broadcast is from "On Optimizing the Communication of Model Parallelism"
 * (section 3.1).
 *
 * Three calls make the path: mv_create (upload a batch of experiments),
 * mv_run (advance every experiment by up to N ticks in one persistent
 * kernel launch), mv_results (per-experiment, per-node and per-message
 * results).  All times are integer ticks; one tick is one packet
 * serialisation time at the experiment's base link rate.
 *
 * Memory: the library never allocates device memory.  The caller gives
 * mv_create a device workspace of at least mv_workspace_bytes() bytes and
 * keeps it alive until mv_destroy.  Host arrays in mv_batch_desc are read
 * during mv_create only.  Every call is bound to the stream given to
 * mv_create; a context is not thread-safe.
 *
 * Errors: every call returns an MV_* status code (negative = error, the
 * context is unchanged unless stated otherwise); mv_strerror names it.
 */
#ifndef MV_H
#define MV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define MV_OK 0              /* every experiment finished (or stopped: OOM,
                                deadlock, overflow)                          */
#define MV_INCOMPLETE 1      /* the tick budget ran out; call mv_run again   */
#define MV_EINVAL (-1)       /* malformed descriptor or argument             */
#define MV_ENOMEM (-2)       /* workspace smaller than mv_workspace_bytes()  */
#define MV_ECUDA (-3)        /* a CUDA call failed (launch, copy, sync)      */
#define MV_ETIMEOUT (-4)     /* the run's watchdog fired: every experiment
                                stopped at a tick boundary (resumable)       */
#define MV_EOVERFLOW (-5)    /* a size or tick count exceeds 32-bit limits   */

/* ---- per-experiment status (mv_results.status) ----------------------- */
#define MV_EXP_DONE 0        /* every DAG node completed                     */
#define MV_EXP_RUNNING 1     /* stopped by the tick budget                   */
#define MV_EXP_OOM 2         /* failed the pre-run GPU memory check          */
#define MV_EXP_DEADLOCK 3    /* nothing in flight, nothing scheduled, not done */
#define MV_EXP_OVERFLOW 4    /* a per-rank table (lanes 64, receive counters
                                128, pending nodes 64, running collectives 16)
                                or a tick value overflowed                   */
#define MV_EXP_ERROR 5       /* unroutable packet or inconsistent schedule   */

/* node kinds, collective kinds and algorithms used in the descriptor */
#define MV_NODE_COMPUTE 0
#define MV_NODE_INTRA 1      /* intra-server collective: alpha + bytes/beta  */
#define MV_NODE_NET 2        /* membership in a network collective           */
#define MV_COLL_ALLREDUCE 0
#define MV_COLL_REDUCESCATTER 1
#define MV_COLL_ALLGATHER 2
#define MV_COLL_RELAY 3      /* pipelined broadcast along the member order   */
#define MV_COLL_P2P 4        /* member 0 sends to member 1                   */
#define MV_COLL_ALLTOALL 5   /* explicit per-pair byte counts                */
#define MV_ALGO_RING 0
#define MV_ALGO_TREE 1       /* all-reduce only; other kinds use the ring    */

#define MV_UNSET 0xFFFFFFFFu /* tick value of "never happened"              */

/*
 * Batch descriptor.  Flat arrays, concatenated over topologies, workloads
 * and experiments in that order.  Indices stored inside a topology's arrays
 * are local to that topology; inside a workload's, local to that workload.
 * All pointers are host pointers, read only during mv_create.
 *
 * Topology t (n_topos of them): topo_nhosts[t] hosts (one NIC each, host h
 * = rank h of any workload run on it), topo_nsw[t] switches, topo_nports[t]
 * switch ports.  Per switch: sw_nports (<= 64), sw_level (1 = edge, higher
 * = closer to the core).  Per port q (switch-major): port_peer[q] >= 0 is
 * the peer switch port, < 0 is host -(peer+1); port_sigma/port_delta
 * describe the link leaving the port (serialisation ticks >= 1, propagation
 * ticks).  Per host: host_port (the switch port it is wired to) and the
 * uplink's host_sigma/host_delta.
 *
 * Workload w: work_nranks[w] ranks; rank_nnodes gives each rank's node
 * count (nodes are numbered rank-major).  Per node: node_kind, node_arg (the
 * collective index for INTRA/NET nodes), node_npred, node_nsucc (successor
 * lists concatenated in succ[], same rank only), node_dur_lo/hi (compute
 * duration in ns; hi > lo draws from [lo, hi] with the experiment's
 * duration seed and node_dur_key).  Per collective: coll_kind, coll_intra
 * (1 = analytic), coll_bytes, coll_nmembers (1..65535), coll_parts (relay partitions
 * K), coll_alpha (ticks, >= 1 for intra), coll_beta_num/den (ticks per
 * byte).  Per member: member_rank, member_node; all-to-all rows
 * (member_a2a_n entries of a2a_dst/a2a_bytes, in rotation order from the
 * next member) and columns (member_a2a_in_n entries of
 * a2a_in_src/a2a_in_bytes).  mem: 10 uint64 per workload: params, tp, pp,
 * layers per stage, micro-batches, seq, batch, hidden, heads, enabled.
 *
 * Experiment e: exp_topo, exp_work, exp_algo, exp_nc (channels, 1..1024),
 * exp_chunk (bytes), exp_pkt (packet bytes), exp_cap (queue slots, 2..1024),
 * exp_tick_ps, exp_dur_seed, exp_ecmp_seed, exp_gpu_mem (bytes per GPU),
 * exp_rec_cap (per-message completion records kept, 0 = none), exp_voq (the
 * switches' ingress buffers: 0 = one FIFO per ingress port, head-of-line
 * blocking kept; 1 = virtual output queues, needs exp_cap <= 64).
 *
 * exp_cc (may be NULL: no congestion control anywhere): MV_CC_FIELDS words
 * per experiment.  [0] selects none (0), DCQCN (1) or DCTCP (2); the
 * Multiverse page, section 5, names both among its congestion-control
 * algorithms.  DCTCP (Alizadeh et al., SIGCOMM 2010): [1] = [2] the marking
 * threshold (arrived packets in the ingress queue a packet leaves), [4] gain
 * shift (1..16), [13] initial window w0 (packets, >= 1), [14] largest window
 * (w0..65535); receivers acknowledge every packet, an overflowing
 * acknowledgement ring is MV_EXP_OVERFLOW.  DCQCN (Zhu et al., SIGCOMM
 * 2015): [1] kmin and [2] kmax (switch marking thresholds, arrived packets
 * in the ingress queue a packet leaves), [3] pmax (marking probability at
 * kmax, units of 2^-16, <= 65536), [4] gain shift (g = 2^-shift, 1..16),
 * [5] N (ticks between a flow's notifications, >= 1), [6] K (alpha timer,
 * ticks, >= 1), [7] T (rate timer, ticks, >= 1), [8] B (byte counter,
 * packets, >= 1), [9] F (fast-recovery events, <= 65535), [10] R_AI, [11]
 * R_HAI, [12] R_min (units of 2^-20 of the line rate, <= 2^20; R_min >= 1),
 * [13..15] zero.  A notification is a packet from the receiver's NIC to
 * the sender's.  Congestion control with exp_voq = 1 is refused (MV_EINVAL).
 * A workload holds fewer than 2^25 - 256 nodes.
 */
#define MV_CC_FIELDS 16
typedef struct mv_batch_desc {
    uint32_t version;                 /* 1 */
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
    const uint32_t *exp_cc;           /* n_exps x MV_CC_FIELDS, or NULL */
} mv_batch_desc;

/*
 * Results, written by mv_results into caller-owned HOST buffers (any
 * pointer may be NULL to skip that field).  Per experiment (n_exps): status
 * (MV_EXP_*), end_tick (latest node end, the iteration time; MV_UNSET if no
 * node ended), now (the experiment's clock: where a budget-stopped one
 * resumes; one past end_tick for one that stopped for good, 0 if no node
 * ended), packets injected, packet-hops
 * (one packet placed on one link), packets delivered, messages delivered,
 * digest (order-independent 64-bit sum over delivered messages of a hash of
 * (sender node, connection key, delivery tick)), rec_count (records
 * produced; only the first exp_rec_cap are kept).  Per node, concatenated
 * over experiments in batch order (sizes from mv_result_sizes): start and
 * end tick.  Per-message records, concatenated in blocks of exp_rec_cap:
 * sender node, 24-bit connection key, delivery tick, in no particular order
 * (Multiverse section 3.1: the network simulator reports each flow's
 * completion to the system simulator).  Per collective instance,
 * concatenated over experiments in batch order (each experiment's block
 * lists its workload's collectives in order; sizes from mv_result_sizes):
 * coll_start, the earliest start tick of its member nodes (MV_UNSET if none
 * started), and coll_end, the latest end tick of its member nodes (MV_UNSET
 * while some member has not ended); the collective's time is coll_end -
 * coll_start, and the iteration time is end_tick.  These are computed on
 * the device from the per-node ticks when either pointer is given.
 */
typedef struct mv_results_view {
    uint32_t *status, *end_tick, *now;
    uint64_t *pkts_injected, *pkt_hops, *pkts_delivered, *msgs_delivered, *digest;
    uint32_t *rec_count;
    uint32_t *node_start, *node_end;
    uint32_t *rec_sender, *rec_key, *rec_tick;
    uint32_t *coll_start, *coll_end;
} mv_results_view;

typedef struct mv_ctx mv_ctx;

/* Options of one mv_run call.
 * watchdog_ns: 0 = none.  Otherwise, once the launch has run that long
 *   (device global timer), every block stops its experiment at the next
 *   tick boundary it checks (every 256 ticks), takes no further experiment,
 *   and mv_run_ex returns MV_ETIMEOUT.  The state stays consistent: a later
 *   mv_run continues where each experiment stopped.  The kernel holds no
 *   lock and waits on no other block, so it cannot hang; the watchdog bounds
 *   the run time of a call.
 * grid_blocks: 0 = every block that fits on the device at once.
 * stage: 0 = an experiment's whole state is staged in shared memory when it
 *   fits, else its hottest arrays in priority order up to the build's share
 *   (wake table, switch and host records, dirty words, queue words, egress
 *   state, up lists, rank control words, port records, running lists);
 *   1 = only its wake table is; 2 = nothing is (results are the same in
 *   every mode; the modes exist to test and measure that).
 * block_warps: warps of the block stepping one experiment (0 = automatic;
 *   at most 8, 16 for variant 3, 32 for variant 4).
 * variant: the kernel build.  0 = automatic; 1 = one block an SM with the
 *   most registers (for batches whose experiments all fit in shared memory);
 *   2 = two 8-warp blocks an SM (more experiments in flight); 3 = one
 *   16-warp block an SM with twice the shared memory for staging (for
 *   experiments whose hottest arrays do not fit variant 2's share); 4 = one
 *   32-warp block an SM at 64 registers a thread (twice the warps stepping
 *   one experiment).  Results are the same in every variant. */
typedef struct mv_run_opts {
    uint64_t watchdog_ns;
    uint32_t grid_blocks;
    uint32_t stage;
    uint32_t block_warps;
    uint32_t variant;
} mv_run_opts;

/* Workspace bytes mv_create needs for this batch (validates the
 * descriptor).  Multiverse section 3.3: the simulator manages the storage
 * of every experiment's entities centrally, one column table per component
 * with an experiment id; here that is one caller-owned device buffer laid
 * out per experiment.  Returns MV_OK, MV_EINVAL or MV_EOVERFLOW. */
int mv_workspace_bytes(const mv_batch_desc *desc, uint64_t *bytes);

/* Sizes of the concatenated per-node, per-record and per-collective result
 * arrays (any pointer may be NULL).  Returns MV_OK or the error of
 * mv_workspace_bytes for this descriptor. */
int mv_result_sizes(const mv_batch_desc *desc, uint64_t *n_nodes, uint64_t *n_records,
                    uint64_t *n_colls);

/* Multiverse section 3.1: the user sets the workload, the collective
 * library's parameters and the topology and lists the experiments; the GPU
 * memory simulator checks each experiment before the run (an experiment
 * that does not fit ends with MV_EXP_OOM).
 * Validate the batch, lay it out in the caller's device workspace
 * (`dev_workspace`, `ws_bytes`, 256-byte aligned), upload it on `stream`
 * (a cudaStream_t, NULL = legacy default stream), build the routing tables,
 * run the memory check and put every experiment at tick 0.  On success
 * *out owns a host-side context (free with mv_destroy); the workspace stays
 * the caller's. */
int mv_create(const mv_batch_desc *desc, void *dev_workspace, uint64_t ws_bytes,
              void *stream, mv_ctx **out);

/* Multiverse section 4.3: one megakernel launch runs the whole execution
 * graph (section 3.2's eight systems in order, every step) for the batch.
 * Advance every unfinished experiment by at most max_ticks ticks of its own
 * clock, in ONE launch of the persistent megakernel, and wait for it.
 * (Ticks are 32-bit: a clock stops at 0xFFF00000, so a larger budget would
 * mean nothing.)  Each
 * experiment is stepped by one thread block (its entities spread over the
 * block's warps, one block barrier per tick); blocks take experiments
 * largest first.  State stays on the device, so run(a) then run(b) equals
 * run(a + b).  *steps_done (may be NULL) receives the largest number of
 * ticks one experiment processed in this call.  Returns MV_OK when no
 * experiment is still running, MV_INCOMPLETE when some hit the budget, or
 * an error. */
int mv_run(mv_ctx *ctx, uint32_t max_ticks, uint64_t *steps_done);
int mv_run_ex(mv_ctx *ctx, uint32_t max_ticks, const mv_run_opts *opts,
              uint64_t *steps_done);

/* Put every experiment back to tick 0 (clear the dynamic state, rebuild the
 * routing tables, rerun the memory check of Multiverse section 3.1) without
 * re-uploading the batch.  Enqueued on the context's stream; does not wait.
 * Returns MV_OK, MV_EINVAL for a NULL context or MV_ECUDA. */
int mv_reset(mv_ctx *ctx);

/* Device time, in ms, of the megakernel launch of the last mv_run, taken
 * with CUDA events recorded on the context's stream around that launch.
 * MV_EINVAL when no run was timed since create or reset. */
int mv_last_run_ms(mv_ctx *ctx, float *ms);

/* Multiverse section 3.1: the network simulator tells the system simulator
 * when each flow completes.  Copy the results (per experiment, per node,
 * per message record, per collective: see mv_results_view) to the caller's
 * host buffers, blocking on the stream.  Returns MV_OK, MV_EINVAL for a
 * NULL context or view, MV_ECUDA if a copy fails. */
int mv_results(mv_ctx *ctx, const mv_results_view *out);

/* Free the host context (and its two CUDA events).  The workspace is not
 * touched and stays the caller's.  MV_EINVAL for NULL. */
int mv_destroy(mv_ctx *ctx);

/*
 * Allocation-free one-shot simulation.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- for
 * example code running inside a framework whose caching allocator already
 * holds the free device memory, a plugin host whose policy forbids new
 * device allocations, or a latency-critical loop where cudaMalloc's implicit
 * device synchronisation is not acceptable.
 *
 * It does what mv_create + mv_run + mv_results + mv_destroy do, but its
 * workspace is a file-scope device array of MV_STATIC_SCRATCH_BYTES (32 MiB)
 * inside the library instead of caller memory.  The caller still passes the
 * batch (host arrays, as for mv_create) and the host result buffers (as for
 * mv_results); `stream` is a cudaStream_t (NULL = legacy default stream),
 * `max_ticks` and `steps_done` are as for mv_run.  It calls no cudaMalloc,
 * cudaFree or other device-allocating routine.
 *
 * The array belongs to the current device: the first call on a device looks
 * up its device address (cudaGetSymbolAddress, with that device current)
 * and keeps it, so make that first call before any stream capture begins.
 * A later call looks the address up again only if the library's device data
 * was re-initialised since (for example after cudaDeviceReset), which it
 * detects by a token it keeps beside the array.  Every call waits for its
 * stream (the results are copied to host memory before it returns).  Once
 * the library's module is loaded on a device, the 32 MiB stay reserved
 * there until the process exits.  Every call reuses the same array (each
 * call clears and re-uploads what it needs), so calls whose GPU work
 * overlaps -- two host threads, or two streams of the same device -- race
 * and must be serialised by the caller.
 *
 * Returns MV_OK / MV_INCOMPLETE as mv_run does, MV_ENOMEM when the batch
 * needs more than MV_STATIC_SCRATCH_BYTES of workspace (see
 * mv_workspace_bytes), or the error of the failing step.
 */
#define MV_STATIC_SCRATCH_BYTES (32ull << 20)
int mv_simulate_static(const mv_batch_desc *desc, uint32_t max_ticks, void *stream,
                       const mv_results_view *out, uint64_t *steps_done);

const char *mv_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* MV_H */
