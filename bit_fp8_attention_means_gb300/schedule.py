"""Amortized grouping schedule over the denoising steps.

Paper summary (paper.rainbus.top), 方法步骤详情 step 1 and 核心方法: cluster
only in the first 25% of the denoising steps, warm-start the centroids from
the previous clustering, and reuse each permutation for 4 neighbouring steps;
dimensionstp.github.io section 3-2 (first-quarter grouping, permutation reuse
in later steps).

Reading used where the pages are silent: a step s clusters when
s < ceil(0.25 * S) and s % 4 == 0; every other step reuses the last
permutation.  The first clustering is a cold start (``cold_iters`` Lloyd
iterations); later ones run ``warm_iters`` iterations from the previous
centroids.  The centroids and pi are the only state carried between steps;
``state_dict`` / ``load_state_dict`` checkpoint and restore it.
"""
import math
from dataclasses import dataclass, field

import torch

from . import vc


def clusters_at(step: int, total_steps: int, quarter: float = 0.25, reuse: int = 4) -> bool:
    return step < math.ceil(quarter * total_steps) and step % reuse == 0


@dataclass
class GroupingState:
    """Cross-step state the caller keeps: centroids, labels and pi."""
    centroids: torch.Tensor = None
    labels: torch.Tensor = None
    perm: torch.Tensor = None
    workspace: torch.Tensor = None
    clusterings: int = 0


def state_dict(state: GroupingState) -> dict:
    """The cross-step state to checkpoint: copies of the centroids, labels and
    pi, and the number of clusterings so far (the workspace is scratch and is
    not kept).  Copies, because later clustering steps write the live tensors
    in place: a checkpoint held in memory stays what it was when taken."""
    def cp(t):
        return None if t is None else t.clone()
    return {"centroids": cp(state.centroids), "labels": cp(state.labels), "perm": cp(state.perm),
            "clusterings": state.clusterings}


def load_state_dict(d: dict, device=None) -> GroupingState:
    """A GroupingState from `state_dict` output, its tensors moved to `device`
    (as saved when None).  The next clustering warm-starts from the restored
    centroids and the steps in between reuse the restored pi, as in an
    uninterrupted run."""
    def mv(t):
        return t if t is None or device is None else t.to(device)
    return GroupingState(centroids=mv(d["centroids"]), labels=mv(d["labels"]), perm=mv(d["perm"]),
                         clusterings=int(d["clusterings"]))


@dataclass
class StepTimes:
    cluster_ms: list = field(default_factory=list)
    quantize_ms: list = field(default_factory=list)
    attn_ms: list = field(default_factory=list)


def run_step(state: GroupingState, Q, K, V, step: int, total_steps: int, k: int, cold_iters: int, warm_iters: int,
             qz=None, O=None, expcast=1, vsmooth=1, times: StepTimes = None, stream=None, force_cluster=False):
    """One denoising step of the hot path: (maybe) group, quantize, attend.

    Returns (qz, O).  When ``times`` is given, CUDA events on the current
    stream time each part (read after a synchronize).
    """
    stream = stream or torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if times is not None else None
    if ev:
        ev[0].record(stream)
    if vsmooth and (force_cluster or clusters_at(step, total_steps) or state.perm is None):
        warm = state.centroids is not None
        state.centroids, state.labels, state.perm = vc.vc_cluster(
            V, k, warm_iters if warm else cold_iters, warm_start=warm, centroids=state.centroids,
            labels=state.labels, perm=state.perm, workspace=state.workspace, stream=stream)
        state.clusterings += 1
    if ev:
        ev[1].record(stream)
    qz = vc.vc_quantize(Q, K, V, state.perm if vsmooth else None, vsmooth, out=qz, stream=stream)
    if ev:
        ev[2].record(stream)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q), expcast=expcast, vsmooth=vsmooth, O=O, stream=stream)
    if ev:
        ev[3].record(stream)
        times._pending = getattr(times, "_pending", []) + [ev]
    return qz, O


def collect(times: StepTimes):
    """Move the recorded events of finished steps into the millisecond lists."""
    for ev in getattr(times, "_pending", []):
        times.cluster_ms.append(ev[0].elapsed_time(ev[1]))
        times.quantize_ms.append(ev[1].elapsed_time(ev[2]))
        times.attn_ms.append(ev[2].elapsed_time(ev[3]))
    times._pending = []
    return times
