"""The oracle's pins are strong enough to catch plausible mistakes: each entry
plants one mistake in a copy of the oracle (an off-by-one, a dropped term, a
wrong index or order, a swapped operand), builds it with gcc, and runs the
pin suite against it (tests/test_oracle_pins.py, through MV_ORACLE_LIB); the
suite must not pass (a pin fails, or the planted mistake crashes the oracle).  Left out, with the reason: a different but equally valid
ECMP hash (the exact hash is a convention, pinned only by GPU = oracle
parity); counting a member that started this very tick as started for an
intra-server completion (equivalent: the completion tick is the same, since
alpha >= 1); reading a queue's current tail instead of its start-of-tick
tail (equivalent: a packet pushed this tick is not ready before the next);
a membership's latest event starting at 0 instead of its join tick
(equivalent: every event comes after the join); a receive queue's credit
delay taken from the uplink instead of the downlink (equivalent on every
fabric here, whose links have one delay both ways); receive counters placed last-fit instead of first-fit (where a
membership's counters sit changes no tick, only which fragmentation first
overflows the table); a zero-byte message of no packets (caught, but it
makes runs very long)."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = [
    ('credit_cap_off_by_one',
     'return s->tail[f] - (h - back) < s->cap;',
     'return s->tail[f] - (h - back) <= s->cap;'),
    ('credit_delay_strict',
     'if (pt + d <= t) break;',
     'if (pt + d < t) break;'),
    ('fwd_drop_delta',
     'p.ready = t + s->port_sigma[qe] + s->port_delta[qe];',
     'p.ready = t + s->port_sigma[qe];'),
    ('ack_hops_drop_one',
     'p.hopsum += s->port_delta[qe] + 1;',
     'p.hopsum += s->port_delta[qe];'),
    ('eg_rr_stays',
     's->eg_rr[qe] = (i + 1) % P;',
     's->eg_rr[qe] = i % P;'),
    ('ring_dep_off_by_one',
     'if (k >= 1) { L->dep_mask = 1u; L->dep_need = (uint32_t)(l * steps + k); }',
     'if (k >= 1) { L->dep_mask = 1u; L->dep_need = (uint32_t)(l * steps + k - 1); }'),
    ('partition_extra_last',
     'return S / nc + (c < S % nc ? 1 : 0);',
     'return S / nc + (c >= nc - S % nc ? 1 : 0);'),
    ('ring_block_sign',
     'uint64_t blk = ((uint64_t)i + N - (k % N)) % N;',
     'uint64_t blk = ((uint64_t)i + (k % N)) % N;'),
    ('relay_no_dep',
     'if (i >= 1) { L->dep_mask = 1u; L->dep_need = m + 1; }',
     'if (i >= 1) { L->dep_mask = 1u; L->dep_need = m; }'),
    ('compute_floor',
     'return (uint32_t)ceil_div(ns * 1000, s->tick_ps);',
     'return (uint32_t)(ns * 1000 / s->tick_ps);'),
    ('intra_ar_factor',
     'case C_AR: be = ceil_div(2 * (g - 1) * S, g); break;',
     'case C_AR: be = ceil_div((g - 1) * S, g); break;'),
    ('edge_zero_cost',
     's->cand[v] = umax32(s->cand[v], c + 1);',
     's->cand[v] = umax32(s->cand[v], c);'),
    ('rdv_no_delay',
     'if (s->start[dnode] == UNSET || s->start[dnode] + s->rdv_delay > t) continue;',
     'if (s->start[dnode] == UNSET || s->start[dnode] > t) continue;'),
    ('inject_no_busy',
     'n->busy = t + s->host_sigma[r];',
     'n->busy = t;'),
    ('nic_rr_stays',
     'n->rr = (q + 1) % NLANE;',
     'n->rr = q;'),
    ('ack_sender_time',
     's->done_max[p.sender] = umax32(s->done_max[p.sender], t + p.hopsum);',
     's->done_max[p.sender] = umax32(s->done_max[p.sender], t);'),
    ('tree_dep_children',
     'L->dep_mask = i == 0 ? child_mask : 1u;',
     'L->dep_mask = 1u;'),
    ('mem_fit_strict',
     'return weights + acts <= cap;',
     'return weights + acts < cap;'),
    ('mem_acts_pp',
     'uint64_t acts = layers * umin(m, pp) * per_layer / tp;',
     'uint64_t acts = layers * m * per_layer / tp;'),
    ('a2a_stripe',
     'uint64_t g = (uint64_t)chan + (uint64_t)m * s->nc;',
     'uint64_t g = (uint64_t)m + (uint64_t)chan * s->nc;'),
    ('same_tick_forward',
     'return p->ready <= t ? p : NULL;',
     'return p->ready < t ? p : NULL;'),
    ('dur_range',
     'if (hi > lo) ns = lo + mix64(mix64((uint64_t)s->node_dur_key[u]) ^ s->dur_seed) % (hi - lo + 1);',
     'if (hi > lo) ns = lo + mix64(mix64((uint64_t)s->node_dur_key[u]) ^ s->dur_seed) % (hi - lo);'),
    ('intra_min_start',
     'else b = umax32(b, st);',
     'else b = b == 0 ? st : (st < b ? st : b);'),
    ('net_done_ignores_acks',
     'complete(s, u, s->done_max[u]);',
     'complete(s, u, t);'),
    ('start_order_reverse',
     'return x < y ? -1 : x > y;',
     'return x > y ? -1 : x < y;'),
    ('lane_slot_highest',
     'for (int q = 0; q < NLANE && slot < 0; q++)',
     'for (int q = NLANE - 1; q >= 0 && slot < 0; q--)'),
    ('tree_parent_port',
     'L->dst_port = chan * 3 + (i == 2 * par + 1 ? 1 : 2);',
     'L->dst_port = chan * 3 + (i == 2 * par + 1 ? 2 : 1);'),
    ('tree_chunk_cap',
     'bytes = P > (uint64_t)m * C ? umin(C, P - (uint64_t)m * C) : 0;',
     'bytes = P > (uint64_t)m * C ? P - (uint64_t)m * C : 0;'),
    ('ring_loops_floor',
     'return P == 0 ? 1 : ceil_div(P, stride);',
     'return P == 0 ? 1 : (P / stride > 0 ? P / stride : 1);'),
    ('ring_steps_ar',
     'return s->coll_kind[c] == C_AR ? 2 * (N - 1) : N - 1;',
     'return s->coll_kind[c] == C_AR ? 2 * N - 1 : N - 1;'),
    ('relay_parts_last',
     'bytes = S / K + (m < S % K ? 1 : 0);',
     'bytes = S / K + (m >= K - S % K ? 1 : 0);'),
    ('p2p_chunk_ignored',
     'bytes = S > (uint64_t)m * C ? umin(C, S - (uint64_t)m * C) : 0;',
     'bytes = S;'),
    ('receive_not_ready',
     'return p->ready <= t ? p : NULL;',
     'return p ? p : NULL;'),
    ('host_delay_drop',
     'p.ready = t + s->host_sigma[r] + s->host_delta[r];',
     'p.ready = t + s->host_sigma[r];'),
    ('host_hop_sum',
     'p.hopsum = s->host_delta[r] + 1;',
     'p.hopsum = s->host_delta[r];'),
    ('rdv_min_delta',
     'if (dl + 1 < s->rdv_delay) s->rdv_delay = dl + 1;\n    }\n    for (uint32_t h = 0;',
     'if (dl + 2 < s->rdv_delay) s->rdv_delay = dl + 2;\n    }\n    for (uint32_t h = 0;'),
    ('deadlock_as_done',
     'if (nx == UNSET) { s->status = ST_DEADLOCK; t++; break; }',
     'if (nx == UNSET) { s->status = ST_DONE; t++; break; }'),
    ('overflow_pend_limit',
     'if (n->n_pend >= NPEND) { fail(s, ST_OVERFLOW); return; }',
     'if (n->n_pend >= NPEND + 1) { fail(s, ST_OVERFLOW); return; }'),
    ('act_limit',
     'if (n->n_act >= NACT) { fail(s, ST_OVERFLOW); return; }',
     'if (n->n_act > NACT) { fail(s, ST_OVERFLOW); return; }'),
    ('memory_weights',
     'uint64_t weights = 16 * params / (tp * pp);',
     'uint64_t weights = 16 * params / tp;'),
    ('digest_drop_tick',
     's->digest += mix64(mix64((uint64_t)p.sender | ((uint64_t)p.key << 32)) ^ (uint64_t)t);',
     's->digest += mix64(mix64((uint64_t)p.sender | ((uint64_t)p.key << 32)));'),
    ('intra_rs_factor',
     'case C_RS: case C_AG: be = ceil_div((g - 1) * S, g); break;',
     'case C_RS: case C_AG: be = ceil_div(g * S, g); break;'),
    ('route_lowest_port_sw',
     'if (s->route[(size_t)w2 * H + h] >= 0 && s->route[(size_t)w * H + h] < 0)',
     'if (s->route[(size_t)w2 * H + h] >= 0)'),
    ('poplog_index',
     'uint32_t pt = s->poplog[(size_t)f * 64 + (h - 1 - back) % 64];',
     'uint32_t pt = s->poplog[(size_t)f * 64 + (h - back) % 64];'),
    ('rr_scan_from_zero',
     'uint32_t i = (s->eg_rr[qe] + k) % P;',
     'uint32_t i = k % P;'),
    ('tree_bcast_child',
     'L->dst_member = 2 * i + L->kind;',
     'L->dst_member = 2 * i + 3 - L->kind;'),
    ('tree_nmsg_root',
     'if (kind == 0) return i > 0 ? (uint32_t)nch : 0;\n            if (kind == 1)',
     'if (kind == 0) return (uint32_t)nch;\n            if (kind == 1)'),
    ('a2a_in_count',
     'tot += n_chunks(s->a2a_in_bytes[e], s->chunk);\n        return (uint32_t)tot;',
     'tot += n_chunks(s->a2a_in_bytes[e], s->chunk);\n        return (uint32_t)tot + 1;'),
    ('due_check_strict',
     'for (int k = 0; k < n->n_pend && !due; k++) due = n->pend_start[k] <= t;',
     'for (int k = 0; k < n->n_pend && !due; k++) due = n->pend_start[k] < t;'),
    ('skip_past_ready',
     'if (rd > t && rd < best) best = rd;',
     'if (rd > t && rd + 1 < best) best = rd + 1;'),
    ('rec_tick_late',
     's->rec_tick[s->rec_count] = t;',
     's->rec_tick[s->rec_count] = t + 1;'),
    ('mem_disabled_check',
     'if (mem[9] == 0) return 1;',
     'if (mem[9] == 0) return 0;'),
    ('ring_last_block_full',
     'bytes = B > blk * bs ? umin(bs, B - blk * bs) : 0;',
     'bytes = bs;'),
    ('relay_dst',
     'L->dst_member = i + 1;\n        L->dst_port = 0;\n        if (i >= 1)',
     'L->dst_member = N - 1;\n        L->dst_port = 0;\n        if (i >= 1)'),
    ('outstanding_recv_only',
     's->outstanding[p.sender]--;',
     '(void)0;'),
    ('tree_kids_left_only',
     'uint32_t child_mask = (has_l ? 2u : 0u) | (has_r ? 4u : 0u);',
     'uint32_t child_mask = (has_l ? 2u : 0u);'),
    ('skip_past_busy',
     'if (n->busy > t && n->busy < best) best = n->busy;',
     'if (n->busy > t && n->busy + 1 < best) best = n->busy + 1;'),
    ('skip_past_credit',
     'if (at < best) best = at;',
     'if (at + 1 < best) best = at + 1;'),
    ('skip_past_eg',
     'if (s->eg_busy[q] > t && s->eg_busy[q] < best) best = s->eg_busy[q];',
     'if (s->eg_busy[q] > t && s->eg_busy[q] + 1 < best) best = s->eg_busy[q] + 1;'),
    ('skip_past_join',
     'best = st + s->rdv_delay;',
     'best = st + s->rdv_delay + 1;'),
    ('skip_past_pend',
     'if (n->pend_start[k] > t && n->pend_start[k] < best) best = n->pend_start[k];',
     'if (n->pend_start[k] > t && n->pend_start[k] + 1 < best) best = n->pend_start[k] + 1;'),
    ('fail_stops_others',
     '        for (uint32_t r = 0; r < s->R; r++)\n            if (!s->nics[r].tick_fail) inject(s, r, t);',
     '        if (s->status != ST_RUNNING) break;\n        for (uint32_t r = 0; r < s->R; r++)\n            if (!s->nics[r].tick_fail) inject(s, r, t);'),
]


def _caught(tmp, name, old, new):
    src = open(O.SRC).read()
    assert src.count(old) == 1, name
    c = os.path.join(tmp, f"{name}.c")
    lib = os.path.join(tmp, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", lib, c])
    env = dict(os.environ, MV_ORACLE_LIB=lib)
    p = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    return name, p.returncode


def test_pins_catch_every_planted_mistake(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        res = list(ex.map(lambda m: _caught(str(tmp_path), *m), MUTANTS))
    survived = [n for n, rc in res if rc == 0]      # the pin suite passed regardless
    assert not survived, f"mutants not caught by the pins: {survived}"
