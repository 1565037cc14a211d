"""Device-resident layers built from the seeded draws of :mod:`synth`.

The F32 draws are made on the host (``synth``) and packed into the int4
container on the GPU by the library's own converter (``pack_int4``).  The
oracle side packs the same draws with its own code; the two never exchange
data.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import synth


def build_device_layer(wl: synth.Workload, layer: int = 0, device: str = "cuda",
                       workers: int | None = None, experts=None, wbits: int = 4):
    """Return a dict of device tensors for one layer:
    router_w [E][H], router_b [E], expert_w4 [E][3FH*wbits/8] uint8, expert_rs [E][2F+H],
    shared_w4 [3FH*wbits/8] uint8, shared_rs [2F+H].

    ``wbits``: the weight container, 4 (packed int4, the library's pack_int4)
    or 8 (int8 codes, pack_int8), packed from the same F32 draw.
    ``experts``: optional iterable of routed expert ids to fill; the others are
    left as zero bytes (used by small tests that know which experts run)."""
    import int4_routed_expert_f32_gb300 as coli

    H, F, E = wl.hidden, wl.ffn, wl.n_experts
    stride = 3 * F * H * wbits // 8
    W, b = synth.router(wl, layer)
    out = dict(
        router_w=torch.from_numpy(W).to(device),
        router_b=torch.from_numpy(b).to(device),
        expert_w4=torch.zeros((E, stride), dtype=torch.uint8, device=device),
        expert_rs=torch.zeros((E, 2 * F + H), dtype=torch.float32, device=device),
        shared_w4=torch.zeros((stride,), dtype=torch.uint8, device=device),
        shared_rs=torch.zeros((2 * F + H,), dtype=torch.float32, device=device),
    )
    ids = list(range(E)) if experts is None else sorted(set(int(e) for e in experts))
    ids = ids + [E]
    staging = torch.empty(3 * F * H, dtype=torch.float32, device=device)

    def pack_into(e, flat):
        staging.copy_(torch.from_numpy(flat), non_blocking=False)
        w4 = out["shared_w4"] if e == E else out["expert_w4"][e]
        rs = out["shared_rs"] if e == E else out["expert_rs"][e]
        mats = ((0, F, H), (F * H, F, H), (2 * F * H, H, F))
        w4off, rsoff = 0, 0
        for off, rows, K in mats:
            nb = rows * K * wbits // 8
            if wbits == 8:
                coli.pack_int8(staging[off:off + rows * K].view(rows, K),
                               w4[w4off:w4off + nb].view(torch.int8).view(rows, K), rs[rsoff:rsoff + rows])
            else:
                coli.pack_int4(staging[off:off + rows * K].view(rows, K),
                               w4[w4off:w4off + nb].view(rows, K // 2), rs[rsoff:rsoff + rows])
            w4off += nb
            rsoff += rows
        torch.cuda.current_stream().synchronize()

    workers = workers or min(16, max(1, (torch.get_num_threads() or 8)))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        futs = [ex.submit(synth.expert_f32_rows, wl, e, layer) for e in ids[:workers]]
        nxt = workers
        for i, e in enumerate(ids):
            flat = futs[i].result()
            if nxt < len(ids):
                futs.append(ex.submit(synth.expert_f32_rows, wl, ids[nxt], layer))
                nxt += 1
            pack_into(e, flat)
            futs[i] = None
    return out
