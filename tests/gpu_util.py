"""GPU-side helpers for the parity tests: move a workloads.Case to the device and run
the library through its C ABI (via the ctypes binding)."""
from __future__ import annotations

import numpy as np


def to_device(case):
    import torch
    dev = torch.device("cuda", 0)

    def conv(x):
        if case.dtype == "bf16":
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    return dict(q_nope=conv(case.q_nope), q_pe=conv(case.q_pe), c_kv=conv(case.c_kv), k_pe=conv(case.k_pe),
                prefix_len=torch.from_numpy(case.prefix_len.astype(np.int32)).to(dev),
                parent=torch.from_numpy(case.parent.astype(np.int32)).to(dev))


def run(case, impl="auto", num_splits=0, vis=None, use_bits=None, max_kv_len=None, dev_tensors=None):
    """Run kdt_verify_attn. ``vis``: caller bits (numpy uint32 [B,T,W]); ``use_bits``: build the bits
    with kdt_build_visibility first and pass them (default: the case's vis_input)."""
    import torch
    import speculative_decoding_tree_absorb_gb300 as kdt
    d = dev_tensors or to_device(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if use_bits is None:
        use_bits = case.vis_input == "bits"
    kw = {}
    if vis is not None:
        kw["vis"] = torch.from_numpy(vis.view(np.int32)).cuda()
    elif use_bits:
        kw["vis"] = kdt.build_visibility(d["parent"], err=err)
    else:
        kw["parent"] = d["parent"]
    out, lse = kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], err=err,
                               scale=case.scale, impl=impl, num_splits=num_splits,
                               max_kv_len=case.max_kv_len if max_kv_len is None else max_kv_len, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), int(err.item())
