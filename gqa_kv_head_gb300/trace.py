"""Timeline of the keys-on-M attention kernel (attn_sw_kernel), from the
global-timer stamps of its FR_TRACE build.

    python -m gqa_kv_head_gb300.trace [--slice-rows 16|32|64] sweep:256:1:65536 [more workloads ...]

Builds the instrumented variant of the library into _build_trace/ (the
library itself has no stamps), runs fused calls of each workload on seeded
synthetic inputs replicated past 2x L2, replayed from a CUDA graph like
bench.py, and prints for the last call: set-up, the launch wait, the Q rows,
per-tile softmax/MMA issue times and the merge phase (microseconds after the
first CTA's set-up; medians over CTAs, and one CTA's tiles). Needs a GPU.
"""
import math
import sys

TRACE_OFFSET = 32 << 20          # FR_TRACE_OFFSET in csrc/fr_trace.cuh
SLOTS = 64


def main(argv):
    import numpy as np
    import torch

    from . import _abi, build
    build.build(trace=True)
    _abi.load(trace=True)
    from . import ops
    import gen

    layout = 2
    slice_rows = None
    if argv and argv[0] == "--slice-rows":
        slice_rows = int(argv[1])
        argv = argv[2:]
    for name in argv:
        w = gen.make_workload(name)
        plan = ops.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, layout=layout, slice_rows=slice_rows,
                                    workspace_bytes=TRACE_OFFSET)
        n_rep = max(2, math.ceil(2 * 135e6 / (4 * w.n_kv * w.hd)))
        reps = [dict(q=torch.from_numpy(w.q()).cuda(), pos=torch.from_numpy(w.pos()).cuda(),
                     k=torch.from_numpy(w.k()).cuda(), v=torch.from_numpy(w.v()).cuda(),
                     mask=None if w.mask() is None else torch.from_numpy(w.mask()).cuda())
                for _ in range(n_rep)]
        n_cta = plan["splits"] * plan["row_slices"]           # every CTA writes SLOTS stamps
        ws = torch.zeros(TRACE_OFFSET + n_cta * SLOTS * 8, dtype=torch.uint8, device="cuda")
        out = torch.empty((w.n_tok, w.n_head, w.hd), device="cuda")
        st = torch.cuda.Stream()

        def call(i):
            r = reps[i % n_rep]
            ops.decode_attn(r["k"], r["v"], w.n_tok, w.n_head, q=r["q"], pos=r["pos"], rope=w.rope,
                            mask=r["mask"], out=out, workspace=ws[:TRACE_OFFSET], stream=st, layout=layout,
                            slice_rows=slice_rows)

        with torch.cuda.stream(st):
            for i in range(4):
                call(i)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(8 * n_rep):
                call(i)
        with torch.cuda.stream(st):
            g.replay()
            g.replay()
        st.synchronize()
        S = n_cta
        tr = ws[TRACE_OFFSET:TRACE_OFFSET + S * SLOTS * 8].view(torch.int64).view(S, SLOTS).cpu().numpy()
        smid = tr[:, 63].copy()
        tr[:, 63] = tr[:, 0]
        rel = (tr - tr[:, 0].min()) / 1000.0
        med = lambda c: float(np.median(rel[:, c]))
        n_tiles = (w.n_kv // plan["splits"] + 127) // 128
        print(f"== {name}: {plan['splits']} splits x {plan['row_slices']} row slices = {S} CTAs, one per SM; "
              f"stamps in us after the first CTA's set-up (graph replay)")
        print(f"set-up done (median) {med(0):.2f}; launch wait over {med(4):.2f}; "
              f"Q in place {med(3):.2f} (rows landed {med(6):.2f}, roped {med(7):.2f})")
        print(f"epilogue (median): row sums {med(57):.2f}, rows stored {med(58):.2f}, fenced and arriving "
              f"{med(59):.2f} (last {rel[:, 59].max():.2f})")
        print(f"every MMA done {rel[:, 1].min():.2f} .. {rel[:, 1].max():.2f}; split states stored "
              f"{rel[:, 56].min():.2f} .. {rel[:, 56].max():.2f}; end {rel[:, 2].min():.2f} .. {rel[:, 2].max():.2f}")
        order = np.argsort(rel[:, 1])
        print("last MMA done, slowest 12 CTAs (cta/sm: us): " + ", ".join(
            f"{int(b)}/{int(smid[b])}: {rel[b, 1]:.2f}" for b in order[::-1][:12]))
        print("fastest 6: " + ", ".join(f"{int(b)}/{int(smid[b])}: {rel[b, 1]:.2f}" for b in order[:6]))
        c = int(np.argsort(rel[:, 2])[S // 2])
        tiles = "  ".join(
            f"t{i}: S {rel[c, 8 + 4 * i + 2]:.2f} softmax {rel[c, 8 + 4 * i]:.2f}-{rel[c, 8 + 4 * i + 1]:.2f} "
            f"PV {rel[c, 8 + 4 * i + 3]:.2f}" for i in range(min(n_tiles, 12)))
        print(f"CTA {c} (median end): {tiles}")
        del reps, g
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main(sys.argv[1:] or ["sweep:256:1:65536"])
