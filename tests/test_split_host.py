"""The host side of the record-range split (sparse_attention_csa2_gb300.shard) on CPU: two
ranks over gloo, each holding half of every sequence's records.  The compute steps are the
oracle's (scores of a range, a range's top-K candidates, the merge of gathered candidates,
per-range attention partials, their log-sum-exp merge with the sink and the inverse
rotation), so what is tested is the orchestration around them: the ranges, visibility
clipped to a range, position offsets, the order of the gathers, the window on one rank.
Every rank must end with the oracle's unsplit layer: the same indices, the same output."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
import synth

N_RECORDS = 2503


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    inp = synth.make_inputs(synth.scaled(synth.WORKLOADS["batched_decode"], B=3, N=N_RECORDS), seed=77)
    # ragged visibility: all records, past the first range only a little, inside the first range
    nv = np.array([N_RECORDS, 1300, 700], np.int32)
    inp["rows"]["n_visible"] = nv
    inp["rows"]["q_pos"] = nv.astype(np.int64)
    inp["rows"]["swa_pos0"] = np.maximum(nv.astype(np.int64) - inp["params"]["W"] + 1, 0)
    return inp


class OracleSteps:
    """The split's compute steps written with the oracle's functions (float64 numpy)."""

    def __init__(self, inp):
        self.inp = inp
        self.p = inp["params"]

    def scores(self, local, n_visible):
        first, count = local["range"]
        rw, lay = self.inp["rows"], self.inp["layers"][0]
        out = np.full((self.p["Bq"], count), -np.inf)
        for r in range(self.p["Bq"]):
            nv = int(n_visible[r])
            if nv:
                keys = O.keys_of(self.inp, int(rw["seq_of_row"][r]), np.arange(first, first + nv))
                out[r, :nv] = O.index_scores(O.bf16_to_f64(lay["q_idx"][r]), lay["w"][r], keys)
        return torch.from_numpy(out)

    def candidates(self, scores, n_visible, K, first):
        s = scores.numpy()
        rows = s.shape[0]
        cs, cp, cc = np.full((rows, K), -np.inf), np.full((rows, K), -1, np.int64), np.zeros(rows, np.int64)
        for r in range(rows):
            sel = O.topk_set(s[r, :int(n_visible[r])], K)
            cs[r, :len(sel)], cp[r, :len(sel)], cc[r] = s[r, sel], first + sel, len(sel)
        return torch.from_numpy(cs), torch.from_numpy(cp), torch.from_numpy(cc)

    def merge(self, scores, pos, cnt, K):
        s, p, c = scores.numpy(), pos.numpy(), cnt.numpy()  # [lists, rows, K_in]
        out = np.full((s.shape[1], K), -1, np.int64)
        for r in range(s.shape[1]):
            sr = np.concatenate([s[l, r, :c[l, r]] for l in range(s.shape[0])])
            pr = np.concatenate([p[l, r, :c[l, r]] for l in range(s.shape[0])])
            sel = np.sort(pr[O.topk_order(sr, K)])  # entry order is position order: ties go low
            out[r, :len(sel)] = sel
        return torch.from_numpy(out)

    def partial(self, local, idx, first, count, skip_window):
        p, rw, lay = self.p, self.inp["rows"], self.inp["layers"][0]
        rows, H, D = p["Bq"], p["H"], p["D"]
        po, pm = np.zeros((rows, 1, H, D)), np.zeros((rows, 1, H, 2))
        pm[..., 0] = -np.inf
        for r in range(rows):
            b, qp = int(rw["seq_of_row"][r]), int(rw["q_pos"][r])
            mine = [int(j) for j in idx[r].numpy() if first <= j < first + count]
            kv = [O.latents_of(self.inp, b, np.array(mine, np.int64))] if mine else []
            if not skip_window:
                kv.append(O.swa_rows_of(self.inp, 0, b, qp))
            if not kv:
                continue
            kv = np.concatenate(kv, 0)
            if kv.shape[0] == 0:
                continue
            z = p["softmax_scale"] * (O.rope(O.bf16_to_f64(lay["q"][r]), qp, p["theta"], p["R"]) @ kv.T)
            m = z.max(axis=1)
            e = np.exp(z - m[:, None])
            po[r, 0] = e @ kv
            pm[r, 0, :, 0], pm[r, 0, :, 1] = m, e.sum(axis=1)
        return torch.from_numpy(po), torch.from_numpy(pm)

    def attn_merge(self, part_o, part_ml, local):
        p, rw, lay = self.p, self.inp["rows"], self.inp["layers"][0]
        po = part_o.numpy().transpose(1, 0, 2, 3, 4).reshape(p["Bq"], -1, p["H"], p["D"])
        pm = part_ml.numpy().transpose(1, 0, 2, 3, 4).reshape(p["Bq"], -1, p["H"], 2)
        out, sm = np.zeros((p["Bq"], p["H"], p["D"])), np.zeros((p["Bq"], p["H"]))
        for r in range(p["Bq"]):
            for h in range(p["H"]):
                m, l, sk = pm[r, :, h, 0], pm[r, :, h, 1], float(lay["sink"][h])
                M = max(float(m.max()), sk)
                f = np.where(np.isfinite(m), np.exp(m - M), 0.0)
                den = float(f @ l) + np.exp(sk - M)
                out[r, h] = (f @ po[r, :, h]) / den
                sm[r, h] = np.exp(sk - M) / den
            out[r] = O.rope(out[r], int(rw["q_pos"][r]), p["theta"], p["R"], sign=-1)
        return torch.from_numpy(out), torch.from_numpy(sm)


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_attention_csa2_gb300.shard import record_ranges, split_full_layer
    inp = _inputs()
    first, count = record_ranges(N_RECORDS, world)[rank]
    local = {"range": (first, count), "n_visible": torch.from_numpy(inp["rows"]["n_visible"])}
    idx, out, sm = split_full_layer(local, first, count, inp["params"]["K"], rank, world, steps=OracleSteps(inp))
    ref = O.csa2_layer(inp, 0)
    results[rank, 0] = float(np.array_equal(idx.numpy(), ref["idx"]))
    results[rank, 1] = float(np.max(np.abs(out.numpy() - ref["o"])) / np.sqrt(np.mean(ref["o"] ** 2)))
    results[rank, 2] = float(np.max(np.abs(sm.numpy() - ref["sink_mass"])))
    dist.barrier()
    dist.destroy_process_group()


def test_record_ranges_cover_every_record_once():
    from sparse_attention_csa2_gb300.shard import record_ranges
    for n, g in ((10, 3), (2503, 2), (1 << 20, 7), (5, 5)):
        rs = record_ranges(n, g)
        assert len(rs) == g and rs[0][0] == 0 and sum(c for _, c in rs) == n
        assert all(a + c == b for (a, c), (b, _) in zip(rs, rs[1:]))
        assert max(c for _, c in rs) - min(c for _, c in rs) <= 1
    with pytest.raises(ValueError):
        record_ranges(3, 4)


def test_split_over_two_gloo_ranks_equals_the_unsplit_layer():
    world, port = 2, _free_port()
    results = torch.zeros(world, 3, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    for rank in range(world):
        assert results[rank, 0] == 1.0, f"rank {rank}: indices differ from the unsplit oracle layer"
        assert results[rank, 1] < 1e-9, f"rank {rank}: output differs by {results[rank, 1]} x RMS"
        assert results[rank, 2] < 1e-12
