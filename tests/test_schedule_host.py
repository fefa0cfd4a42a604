"""Host logic of the amortized grouping schedule (no GPU).

Paper summary (paper.rainbus.top), 方法步骤详情 step 1: cluster only in the
first quarter of the denoising steps, warm-started from the previous
centroids, and reuse a permutation for 4 neighbouring steps.  The checks:

* the steps that cluster, for step counts where the ceiling matters;
* a step sequence through ``run_step`` with the library calls replaced by a
  recorder: the first clustering is cold, later ones warm from the centroids
  the previous one returned, every other step quantizes with the last pi,
  ``vsmooth = 0`` never clusters and quantizes with the identity;
* checkpoint and resume: a run saved after any step and restored from the
  saved bytes makes the same calls as the uninterrupted run.
"""
import math

import pytest

from bit_fp8_attention_means_gb300 import schedule


@pytest.mark.parametrize("S,want", [(50, [0, 4, 8, 12]), (4, [0]), (1, [0]), (16, [0]),
                                    (17, [0, 4]), (20, [0, 4]), (33, [0, 4, 8]), (0, [])])
def test_clustering_steps(S, want):
    got = [s for s in range(S) if schedule.clusters_at(s, S)]
    assert got == want
    # every clustering step lies in the first quarter, rounded up
    assert all(s < math.ceil(0.25 * S) for s in got)


class _Recorder:
    """Stands in for the binding: records each call and returns tokens."""

    def __init__(self):
        self.calls = []
        self.n = 0

    def vc_cluster(self, V, k, iters, warm_start=False, centroids=None, labels=None, perm=None,
                   workspace=None, stream=None):
        self.n += 1
        self.calls.append(("cluster", iters, warm_start, centroids))
        return ("C%d" % self.n, "z%d" % self.n, "pi%d" % self.n)

    def vc_quantize(self, Q, K, V, perm, vsmooth, out=None, stream=None):
        self.calls.append(("quantize", perm, vsmooth))
        return "qz"

    def vc_attn_fwd(self, qz, shape, expcast=1, vsmooth=1, O=None, stream=None):
        self.calls.append(("attn", expcast, vsmooth))
        return "O"

    def shape_of(self, Q):
        return None


def _run(monkeypatch, S, vsmooth=1):
    rec = _Recorder()
    monkeypatch.setattr(schedule, "vc", rec)
    st = schedule.GroupingState()
    for s in range(S):
        schedule.run_step(st, "Q", "K", "V", s, S, k=8, cold_iters=5, warm_iters=1, vsmooth=vsmooth,
                          stream=object())
    return rec, st


def test_step_sequence_cold_then_warm(monkeypatch):
    rec, st = _run(monkeypatch, 50)
    clus = [c for c in rec.calls if c[0] == "cluster"]
    assert [c[1:3] for c in clus] == [(5, False), (1, True), (1, True), (1, True)]
    # each warm start takes the centroids the previous clustering returned
    assert [c[3] for c in clus] == [None, "C1", "C2", "C3"]
    assert st.clusterings == 4 and st.perm == "pi4"
    # the permutation each step quantizes with: the last one computed
    perms = [c[1] for c in rec.calls if c[0] == "quantize"]
    want = ["pi%d" % (min(s // 4, 3) + 1) for s in range(50)]
    assert perms == want
    assert sum(c[0] == "attn" for c in rec.calls) == 50


def test_vsmooth_off_never_clusters(monkeypatch):
    rec, st = _run(monkeypatch, 12, vsmooth=0)
    assert not [c for c in rec.calls if c[0] == "cluster"]
    assert all(c[1] is None and c[2] == 0 for c in rec.calls if c[0] == "quantize")
    assert st.clusterings == 0


def test_missing_permutation_forces_a_clustering(monkeypatch):
    """A state with no pi yet clusters even on a reuse step."""
    rec = _Recorder()
    monkeypatch.setattr(schedule, "vc", rec)
    st = schedule.GroupingState()
    schedule.run_step(st, "Q", "K", "V", 7, 50, k=8, cold_iters=5, warm_iters=1, stream=object())
    assert rec.calls[0][:3] == ("cluster", 5, False)
    assert rec.calls[1] == ("quantize", "pi1", 1)


def test_resume_from_checkpoint_matches_uninterrupted(monkeypatch):
    import io

    import torch
    S = 50
    full, _ = _run(monkeypatch, S)
    for cut in (3, 4, 6, 13):
        rec = _Recorder()
        monkeypatch.setattr(schedule, "vc", rec)
        st = schedule.GroupingState()
        for s in range(cut):
            schedule.run_step(st, "Q", "K", "V", s, S, k=8, cold_iters=5, warm_iters=1, stream=object())
        # the state round-trips through bytes (tensor-valued in real use)
        st.centroids, st.labels, st.perm = (torch.full((2,), float(st.clusterings)),
                                            torch.zeros(3, dtype=torch.int32), torch.arange(3, dtype=torch.int32))
        buf = io.BytesIO()
        torch.save(schedule.state_dict(st), buf)
        buf.seek(0)
        st2 = schedule.load_state_dict(torch.load(buf), device="cpu")
        assert st2.clusterings == st.clusterings
        assert torch.equal(st2.centroids, st.centroids) and torch.equal(st2.perm, st.perm)
        marker = st2.perm
        ncut = len(rec.calls)
        for s in range(cut, S):
            schedule.run_step(st2, "Q", "K", "V", s, S, k=8, cold_iters=5, warm_iters=1, stream=object())
        kinds = [c[0] for c in rec.calls]
        assert kinds == [c[0] for c in full.calls]
        # the first clustering after the resume warm-starts from the restored centroids,
        # and the steps before it quantize with the restored pi
        after = rec.calls[ncut:]
        first = next((i for i, c in enumerate(after) if c[0] == "cluster"), None)
        if first is not None:
            assert after[first][1:3] == (1, True) and torch.equal(after[first][3], st.centroids)
        pre = after[:first] if first is not None else after
        assert all(c[1] is marker for c in pre if c[0] == "quantize")


def test_in_memory_checkpoint_is_not_changed_by_later_steps(monkeypatch):
    """A checkpoint kept in memory (not serialized) is a copy: a later
    clustering that writes the live tensors in place leaves it as taken, and a
    resume from it matches the state at the cut."""
    import torch

    class InPlace(_Recorder):
        def vc_cluster(self, V, k, iters, warm_start=False, centroids=None, labels=None, perm=None,
                       workspace=None, stream=None):
            self.n += 1
            self.calls.append(("cluster", iters, warm_start, centroids))
            if centroids is None:
                return torch.zeros(4), torch.zeros(3, dtype=torch.int32), torch.arange(3, dtype=torch.int32)
            centroids.add_(1.0)        # the device call updates its arguments in place
            labels.add_(1)
            perm.copy_(perm.flip(0))
            return centroids, labels, perm

    rec = InPlace()
    monkeypatch.setattr(schedule, "vc", rec)
    st = schedule.GroupingState()
    schedule.run_step(st, "Q", "K", "V", 0, 50, k=8, cold_iters=5, warm_iters=1, stream=object())
    ck = schedule.state_dict(st)
    at_cut = (st.centroids.clone(), st.labels.clone(), st.perm.clone())
    schedule.run_step(st, "Q", "K", "V", 4, 50, k=8, cold_iters=5, warm_iters=1, stream=object())
    assert not torch.equal(st.centroids, at_cut[0])          # the live state moved on
    for got, want in zip((ck["centroids"], ck["labels"], ck["perm"]), at_cut):
        assert torch.equal(got, want)
    st2 = schedule.load_state_dict(ck)
    assert torch.equal(st2.centroids, at_cut[0]) and torch.equal(st2.perm, at_cut[2]) and st2.clusterings == 1
