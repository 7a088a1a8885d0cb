"""Ragged input order: the per-expert TMA descriptors that the schedule kernel builds on the
device must be byte-identical to descriptors encoded on the host for the same expert blocks
(K-major A: [hidden, n_e] row-major at element begin_e*hidden; K-major B: [intermediate, n_e] at
begin_e*intermediate). Only the schedule kernel runs here; no descriptor is used for a copy."""
import numpy as np
import pytest
import torch

import workloads as W
from kgw_testlib import Outputs, ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("b_major", ["mn", "k"])
@pytest.mark.parametrize("counts,H,I", [
    ([256, 0, 768, 512], 128, 256),           # blocks on both sides of 128 KiB
    ([256, 512, 256, 1024, 0, 2048, 256], 128, 256),
    ([256, 512, 768], 256, 512),
    ([4096, 256, 0, 0, 1280], 384, 512),
    (list(W.counts_zipf(4, 128, 262144, 1.2)), 2048, 768),
])
def test_device_built_descriptors_match_host_encoding(counts, H, I, b_major):
    kgw = ensure_built()
    counts = np.asarray(counts, dtype=np.int64)
    T = int(counts.sum())
    offsets = np.cumsum(counts).astype(np.int32)
    a = torch.empty(H * T, dtype=torch.bfloat16, device=DEV)
    b = torch.empty((T, I), dtype=torch.bfloat16, device=DEV)
    off_d = torch.from_numpy(offsets).to(DEV)
    out = torch.empty((len(counts), H, I), dtype=torch.float32, device=DEV)
    args = kgw.make_args(len(counts), H, I, T, a, b, off_d, out=out, input_order=kgw.KGW_RAGGED,
                         b_major=kgw.KGW_K_MAJOR if b_major == "k" else kgw.KGW_MN_MAJOR)
    ws = kgw.workspace_for(args, device=DEV)
    dump = np.zeros(len(counts) * 512, dtype=np.uint8)
    mism = kgw.kgw_debug_check_ragged_maps(args, False, offsets, ws, host_dump=dump)
    if mism != 0:
        d = dump.reshape(len(counts), 2, 2, 128)
        msgs = []
        for e in np.nonzero(counts)[0]:
            for op in range(2):
                diff = np.nonzero(d[e, op, 0] != d[e, op, 1])[0]
                if len(diff):
                    msgs.append(f"expert {e} operand {'AB'[op]} (n={counts[e]}) bytes {diff.tolist()}: device "
                                f"{d[e, op, 0][diff].tolist()} host {d[e, op, 1][diff].tolist()}")
        pytest.fail(f"{mism} descriptors differ; " + "; ".join(msgs[:4]))
