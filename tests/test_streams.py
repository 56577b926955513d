"""Persistent forwards on several streams at once: each stream's launches hand
out their work items from that stream's own counter pair, so launches that
run concurrently on different streams neither share nor reset each other's
counters.  The outputs must equal, bit for bit, those of the same calls made
one at a time (the forward is deterministic)."""
import numpy as np
import pytest
import torch

import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import inputs

pytestmark = pytest.mark.gpu

PROBLEMS = [  # B, Hq, Hkv, N, d, causal: all with more than 128 rows (the persistent kernel)
    (1, 4, 2, 1000, 128, True),
    (2, 2, 2, 700, 64, False),
    (1, 8, 8, 513, 128, False),
]


def _tensors(i, B, Hq, Hkv, N, d):
    dev = torch.device("cuda", 0)
    out = []
    for k, (h, name) in enumerate(((Hq, "Q"), (Hkv, "K"), (Hkv, "V"))):
        a = inputs.make_tensor(0x57E0 + 16 * i + k, (B, h, N, d), "bf16")
        out.append(torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
    return out


def test_persistent_forward_on_concurrent_streams():
    data = [_tensors(i, *pr[:5]) for i, pr in enumerate(PROBLEMS)]
    ref = []
    for (Q, K, V), pr in zip(data, PROBLEMS):
        ref.append(pkg.attn_fwd(Q, K, V, None, pr[5]))
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in PROBLEMS]
    reps = 6
    outs = []
    torch.cuda.synchronize()
    for _ in range(reps):
        for (Q, K, V), pr, st in zip(data, PROBLEMS, streams):
            with torch.cuda.stream(st):
                outs.append(pkg.attn_fwd(Q, K, V, None, pr[5]))
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    for r in range(reps):
        for j in range(len(PROBLEMS)):
            O, L = outs[r * len(PROBLEMS) + j]
            assert torch.equal(O, ref[j][0]) and torch.equal(L, ref[j][1]), (r, j)
