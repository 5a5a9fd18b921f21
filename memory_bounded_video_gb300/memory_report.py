"""Peak activation memory of the bounded block against sequence length.

    python -m memory_bounded_video_gb300.memory_report [--D 3072 --heads 24
        --ffn 8192 --chunk 4096 --ffn-slice 2048 --T 8192,16384,32768,65536]

For each T: the analytic workspace (dit_block_workspace_bytes), its split
into the K/V floor (4*T*D bytes, which grows with T) and the chunk-bounded
rest, and - with a GPU - the measured device memory the forward needs beyond
the inputs and weights (torch's peak allocation while a plan's workspace is
allocated and the forward runs; the library allocates nothing itself).  The
unchunked reference point is the same plan with chunk 0 and no FFN slicing.
With ``--kv-offload B`` the same is reported for the K/V offload schedule
(K/V in pinned host memory, streamed back in key blocks of B tokens), whose
workspace has no K/V floor.
"""

from __future__ import annotations

import argparse
import json
import sys

from . import ditstream as ds


def analytic(T, D, H, F, chunk, fs, kv_offload=0):
    p = ds.block_plan(T, D, H, F, chunk, chunk, fs)
    full = ds.block_plan(T, D, H, F, 0, 0, 0).workspace_bytes()
    if kv_offload:
        p.set_kv_offload(kv_offload)
        ws = p.workspace_bytes()
        return dict(T=T, workspace=ws, kv_floor=0, rest=ws, unchunked_workspace=full,
                    host_kv=p.kv_host_bytes())
    ws = p.workspace_bytes()
    return dict(T=T, workspace=ws, kv_floor=4 * T * D, rest=ws - 4 * T * D,
                unchunked_workspace=full)


def measured(T, D, H, F, chunk, fs, kv_offload=0):
    import torch

    from . import runner, synth
    inp = synth.make_inputs(T, D, H, F, seed=0)
    dev = runner.upload(inp)
    x = dev.x.clone()
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    stack = runner.DitStack(T, D, H, F, chunk, chunk, fs, kv_offload=kv_offload)
    stack.forward(x, dev)
    stack.check()
    peak = torch.cuda.max_memory_allocated() - base
    del stack
    return peak


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--D", type=int, default=3072)
    ap.add_argument("--heads", type=int, default=24)
    ap.add_argument("--ffn", type=int, default=8192)
    ap.add_argument("--chunk", type=int, default=4096)
    ap.add_argument("--ffn-slice", type=int, default=2048)
    ap.add_argument("--T", default="8192,16384,32768,65536")
    ap.add_argument("--kv-offload", type=int, default=0,
                    help="key block size of the K/V offload schedule (0: K/V resident)")
    ap.add_argument("--measure", action="store_true",
                    help="also run the forward on the GPU and measure")
    a = ap.parse_args(argv)
    ds.load()
    for T in [int(t) for t in a.T.split(",")]:
        r = analytic(T, a.D, a.heads, a.ffn, a.chunk, a.ffn_slice, a.kv_offload)
        if a.measure:
            r["measured_peak"] = measured(T, a.D, a.heads, a.ffn, a.chunk, a.ffn_slice,
                                          a.kv_offload)
        r = {k: (round(v / 2**20, 2) if k != "T" else v) for k, v in r.items()}
        print(json.dumps(dict(unit="MiB", **r)))
    return 0


if __name__ == "__main__":
    sys.exit(main())
