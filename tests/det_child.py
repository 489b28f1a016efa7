"""Digests of one seeded fwd+bwd per case, printed as JSON (run in a separate
process by tests/test_gpu_determinism.py)."""
import hashlib
import json
import sys

import numpy as np


def digests():
    import torch

    import bwd_gn3d_stats_gb300 as gn
    from bwd_gn3d_stats_gb300 import synth

    prev = gn.use_library("testing")  # the launch-form setting is a testing-build hook
    out = {}
    cases = [("ncdhw_stream", (1, 32, 24, 24, 24, 8, synth.BF16), gn.PATH_STREAMING, False),
             ("ncdhw_fused", (1, 32, 24, 24, 24, 8, synth.BF16), gn.PATH_FUSED, False),
             ("ncdhw_f32", (2, 16, 16, 16, 16, 4, synth.F32), gn.PATH_AUTO, False),
             ("ndhwc", (1, 48, 13, 11, 7, 8, synth.BF16), gn.PATH_AUTO, True),
             ("ndhwc_512", (1, 512, 4, 4, 5, 8, synth.BF16), gn.PATH_AUTO, True),
             ("ncdhw_128", (1, 32, 128, 128, 128, 8, synth.BF16), gn.PATH_AUTO, False)]
    for name, shape, path, cl in cases:
        gn.gn3d_debug_set(gn.DEBUG_PATH, path)
        site = synth.Site(*shape)
        inp = synth.make_inputs(site, seed=21)
        dt = torch.bfloat16 if site.dtype == synth.BF16 else torch.float32

        def dev(a):
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
            t = t.view(dt) if a.dtype == np.uint16 else t
            t = t.reshape(site.N, site.C, site.D, site.H, site.W)
            return t.contiguous(memory_format=torch.channels_last_3d) if cl else t

        x, dy = dev(inp["x"]), dev(inp["dy"])
        g, b = torch.from_numpy(inp["gamma"]).cuda(), torch.from_numpy(inp["beta"]).cuda()
        fwd, bwd = (gn.forward_ndhwc, gn.backward_ndhwc) if cl else (gn.forward, gn.backward)
        y, m, r = fwd(x, g, b, site.G)
        dx, dg, db = bwd(dy, x, m, r, g, site.G)
        torch.cuda.synchronize()
        h = hashlib.sha256()
        for t in (y, m, r, dx, dg, db):
            h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
        out[name] = h.hexdigest()
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_AUTO)
    gn.use_library(prev)
    return out


if __name__ == "__main__":
    print(json.dumps(digests()))
    sys.stdout.flush()
