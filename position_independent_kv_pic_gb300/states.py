"""Host driver of the linear-layer state composition (HYPIC blog, section 2.1).

Holds the cached (T_c, S_c) pool of a hybrid model's linear-attention layer on the
device, each request's chain of pool entries, the workspace and the output, and
calls ``pic_compose_states``.  Bookkeeping only: the composition runs in the
library's kernels.
"""

from __future__ import annotations

import numpy as np
import torch

from . import pic_compose_segment, pic_compose_split_t, pic_compose_states, pic_compose_workspace


class ComposeBatch:
    """``T``, ``S``: [n_pool][H][d][d] float32 tensors; ``chains``: per request, the
    pool entries of its linked chunks in link order.  ``seg`` None picks the
    level-0 segment that fills one wave of the device's SMs.  T is cached in the
    split form the kernel reads (two bf16 planes), written once here."""

    def __init__(self, T, S, chains, device="cuda", seg=None):
        assert T.shape == S.shape and T.dim() == 4 and T.shape[2] == T.shape[3]
        self.device = torch.device(device)
        self.n_pool, self.H, self.d = int(T.shape[0]), int(T.shape[1]), int(T.shape[2])
        t32 = T.to(self.device, torch.float32).contiguous()
        self.T = torch.empty((self.n_pool, self.H, 2, self.d, self.d), dtype=torch.bfloat16, device=self.device)
        pic_compose_split_t(t32, self.T)
        del t32
        self.S = S.to(self.device, torch.float32).contiguous()
        lens = np.array([len(c) for c in chains], np.int64)
        off = np.zeros(len(chains) + 1, np.int32)
        off[1:] = np.cumsum(lens)
        flat = np.concatenate([np.asarray(c, np.int32) for c in chains]) if len(chains) else np.zeros(0, np.int32)
        self.chains = [np.asarray(c, np.int32) for c in chains]
        self.n_req = len(chains)
        self.n_elems = int(off[-1])
        self.max_chain = int(lens.max()) if len(lens) else 0
        self.ids = torch.from_numpy(flat if len(flat) else np.zeros(1, np.int32)).to(self.device)
        self.chain_off = torch.from_numpy(off).to(self.device)
        sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.seg = (pic_compose_segment(self.n_req, self.n_elems, self.max_chain, self.H, sms)
                    if seg is None else int(seg))
        ws = pic_compose_workspace(self.n_req, self.max_chain, self.H, self.d, self.seg)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)
        self.out = torch.empty(self.n_req, self.H, self.d, self.d, dtype=torch.float32, device=self.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)

    def run(self, stream=None):
        pic_compose_states(self.T, self.S, self.ids, self.chain_off, self.n_req, self.n_elems, self.max_chain,
                           self.H, self.d, self.seg, self.out, self.ws, self.err, stream)
        return self.out

    def error(self) -> int:
        return int(self.err.item())

    @property
    def launches(self) -> int:
        """Kernel launches of one call: level 0, level 1 (two levels) and, above 352
        requests, the planner (with fewer the CTAs find their work themselves)."""
        if self.n_req == 0:
            return 0
        levels = 1 if (self.seg <= 1 or self.seg >= self.max_chain) else 2
        return levels + (1 if self.n_req > 352 else 0)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes a composition must move: S of every chain element, T of every element
        but the first of each chain, and the output state of every chain."""
        mat = self.d * self.d * 4
        nonempty = sum(1 for c in self.chains if len(c))
        return (2 * self.n_elems - nonempty + self.n_req) * self.H * mat


def _main():
    """Run the composition on a seeded preset's chunk chains and print one JSON line
    (mean time of the timed runs, algorithmic bytes, GB/s)."""
    import argparse
    import json

    from . import build, inputs

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="long_context_100x1000", choices=sorted(inputs.PRESETS))
    ap.add_argument("--heads", type=int, default=32)
    ap.add_argument("--seg", type=int, default=None, help="level-0 segment (default: one wave of SMs)")
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--runs", type=int, default=2)
    a = ap.parse_args()
    build.build()
    wl = inputs.PRESETS[a.workload]()
    T, S, chains = inputs.linear_states(wl, H=a.heads, d=128)
    b = ComposeBatch(T, S, chains, seg=a.seg)
    for _ in range(a.warmup):
        b.run()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.runs)]
    for e0, e1 in ev:
        e0.record()
        b.run()
        e1.record()
    torch.cuda.synchronize()
    if b.error():
        raise SystemExit(f"device error {b.error()}")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / max(len(ev), 1)
    print(json.dumps({"workload": a.workload, "heads": a.heads, "seg": b.seg, "launches": b.launches,
                      "ms": ms, "bytes": b.algorithmic_bytes, "GB/s": b.algorithmic_bytes / (ms / 1e3) / 1e9}))


if __name__ == "__main__":
    _main()
