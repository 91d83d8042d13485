"""Timelines of the decode attention kernels, from the global-timer stamps of
their FR_TRACE build.

    python -m gqa_kv_head_gb300.trace [--layout 1|2] [--slice-rows 16|32|64] sweep:256:1:65536 [more ...]

--layout 2 (the default) traces the keys-on-M kernel (attn_sw_kernel),
--layout 1 the 128-row kernel (attn_tc_kernel) and its merge kernel. Builds
the instrumented variant of the library into _build_trace/ (the library
itself has no stamps), runs fused calls of each workload on seeded synthetic
inputs replicated past 2x L2, replayed from a CUDA graph like bench.py, and
prints for the last call: set-up, the launch wait, the Q rows, per-tile
times and the merge phase (microseconds after the first CTA's set-up;
medians over CTAs). Needs a GPU.
"""
import math
import sys

TRACE_OFFSET = 32 << 20          # FR_TRACE_OFFSET in csrc/fr_trace.cuh
SLOTS = 64
TRACE_CTAS = 2048                # attention CTAs 0..1023, merge-kernel CTAs at 1024 + b


def _run(w, layout, slice_rows, plan, torch):
    from . import ops
    n_rep = max(2, math.ceil(2 * 135e6 / (4 * w.n_kv * w.hd)))
    reps = [dict(q=torch.from_numpy(w.q()).cuda(), pos=torch.from_numpy(w.pos()).cuda(),
                 k=torch.from_numpy(w.k()).cuda(), v=torch.from_numpy(w.v()).cuda(),
                 mask=None if w.mask() is None else torch.from_numpy(w.mask()).cuda())
            for _ in range(n_rep)]
    ws = torch.zeros(TRACE_OFFSET + TRACE_CTAS * SLOTS * 8, dtype=torch.uint8, device="cuda")
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
    tr = ws[TRACE_OFFSET:].view(torch.int64).view(TRACE_CTAS, SLOTS).cpu().numpy()
    del reps, g
    torch.cuda.empty_cache()
    return tr


def _keys_on_m(name, w, plan, tr, np):
    S = plan["splits"] * plan["row_slices"]
    tr = tr[:S].copy()
    smid = tr[:, 63].copy()
    tr[:, 63] = tr[:, 0]
    rel = (tr - tr[:, 0].min()) / 1000.0
    med = lambda c: float(np.median(rel[:, c]))
    n_tiles = (w.n_kv // plan["splits"] + 127) // 128
    print(f"== {name}: keys-on-M kernel, {plan['splits']} splits x {plan['row_slices']} row slices = {S} CTAs, "
          f"one per SM; stamps in us after the first CTA's set-up (graph replay)")
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


def _row_tiles(name, w, plan, tr, np):
    S = plan["row_tiles"] * plan["splits"]
    A = tr[:min(S, 1024)].copy()
    smid = A[:, 63].copy()
    A[:, 63] = A[:, 0]
    t0 = A[:, 0].min()
    rel = (A - t0) / 1000.0
    q = lambda c: f"{rel[:, c].min():.2f}/{np.median(rel[:, c]):.2f}/{rel[:, c].max():.2f}"
    print(f"== {name}: 128-row kernel, {plan['row_tiles']} row tiles x {plan['splits']} splits = {S} CTAs, "
          f"merge kernel {bool(plan['merge_kernel'])}; stamps in us after the first CTA's set-up "
          f"(graph replay; min/median/max over CTAs)")
    print(f"set-up {q(0)}; launch wait over {q(4)}; Q in place {q(3)}")
    for i in range(7):
        has = A[:, 8 + 4 * i] > 0                    # the CTAs with a tile i
        if has.sum() * 2 < len(A):
            break
        md = lambda c: float(np.median(rel[has, c]))
        print(f"  tile {i} ({int(has.sum())} CTAs): K landed {md(36 + i):6.2f}  S issued {md(8 + 4 * i + 2):6.2f}  "
              f"softmax {md(8 + 4 * i):6.2f}-{md(8 + 4 * i + 1):6.2f}  "
              f"P and V ready {md(44 + i):6.2f}  PV issued {md(8 + 4 * i + 3):6.2f}")
    print(f"every MMA done {q(1)}; loop drained {q(57)}; split state stored {q(58)}; end {q(2)}")
    if plan["merge_kernel"]:
        Mg = tr[1024:]
        Mg = Mg[Mg[:, 0] > 0]
        m = (Mg[:, :3] - t0) / 1000.0
        per_sm = np.bincount(Mg[:, 63].astype(np.int64))
        print(f"merge kernel: {len(Mg)} CTAs on {int((per_sm > 0).sum())} SMs (at most {int(per_sm.max())} per SM); "
              f"resident {np.median(m[:, 0]):.2f} (first {m[:, 0].min():.2f}, last {m[:, 0].max():.2f}); "
              f"launch wait over {m[:, 1].min():.2f}/{np.median(m[:, 1]):.2f}; "
              f"end {m[:, 2].min():.2f}/{np.median(m[:, 2]):.2f}/{m[:, 2].max():.2f}")
    order = np.argsort(rel[:, 2])
    print("last to end (cta/sm: us): " + ", ".join(f"{int(b)}/{int(smid[b])}: {rel[b, 2]:.2f}"
                                                  for b in order[::-1][:8]))


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
    while argv and argv[0] in ("--slice-rows", "--layout"):
        if argv[0] == "--slice-rows":
            slice_rows = int(argv[1])
        else:
            layout = int(argv[1])
        argv = argv[2:]
    if layout not in (1, 2):
        raise SystemExit("--layout takes 1 (128-row kernel) or 2 (keys-on-M kernel)")
    for name in argv:
        w = gen.make_workload(name)
        plan = ops.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, layout=layout, slice_rows=slice_rows,
                                    workspace_bytes=TRACE_OFFSET)
        tr = _run(w, layout, slice_rows, plan, torch)
        if layout == 2:
            _keys_on_m(name, w, plan, tr, np)
        else:
            _row_tiles(name, w, plan, tr, np)


if __name__ == "__main__":
    main(sys.argv[1:] or ["sweep:256:1:65536"])
