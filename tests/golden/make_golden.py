"""Write the regression fixtures in this folder.

The pages print no worked example, so every stored value here is written by
this script, which calls only the CPU oracle (``oracle``) on inputs from the
seeded generator (``synth``).  The inputs are stored beside the expected
outputs, so the fixtures do not depend on the host's libm.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def _dump(f, name, a):
    a = np.asarray(a)
    if a.dtype == np.float32:
        vals = " ".join(f"{v:08x}" for v in a.reshape(-1).view(np.uint32))
        kind = "f32hex"
    else:
        vals = " ".join(str(int(v)) for v in a.reshape(-1))
        kind = str(a.dtype)
    f.write(f"{name} {kind} {','.join(map(str, a.shape))} {vals}\n")


def linear_chain_8x64x32(path):
    wl = synth.CONFIGS["linear_chain_8x64x32"]
    d, p = wl.dims, wl.params
    x, w, ws, b = synth.linear_inputs(wl.seed, d["M"], d["K"], d["N"], x_kind="fp32", p=p)
    xq = oracle.quantize_per_tensor(x, p["in_scale"], p["in_zp"])
    out = oracle.linear(xq, p["in_scale"], p["in_zp"], w, ws, b, p["out_scale"], p["out_zp"])
    acc = oracle.linear_acc(xq, p["in_zp"], w)
    with open(path, "w") as f:
        f.write("# quantize_per_tensor -> q8ta_linear, M=8 K=64 N=32, seed 0 (written by "
                "make_golden.py from the CPU oracle)\n")
        f.write(f"# in_scale={p['in_scale']} in_zp={p['in_zp']} out_scale={p['out_scale']} "
                f"out_zp={p['out_zp']}\n")
        for name, a in (("x", x), ("w", w), ("ws", ws), ("b", b), ("xq", xq), ("acc", acc),
                        ("out", out)):
            _dump(f, name, a)


def conv_t_small(path):
    d = dict(N=1, IC=3, H_in=5, W_in=4, OC=4, Kh=3, Kw=3, s=2, p=1, op=1)
    p = dict(in_scale=0.02, in_zp=-7, ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1,
             out_scale=0.15, out_zp=2)
    x, w, ws, b = synth.conv_t_inputs(1234, d, p)
    H, W = synth.output_hw(d["H_in"], d["W_in"], 3, 3, 2, 2, 1, 1, 1, 1)
    acc = oracle.conv2d_transposed_acc(x, p["in_zp"], w, 3, 3, H, W, (2, 2), (1, 1))
    out = oracle.conv2d_transposed(x, p["in_scale"], p["in_zp"], w, 3, 3, ws, b, p["out_scale"],
                                   p["out_zp"], H, W, (2, 2), (1, 1))
    with open(path, "w") as f:
        f.write("# q8ta_conv2d_transposed N=1 IC=3 5x4 OC=4 K=3 s=2 p=1 op=1 -> "
                f"{H}x{W}, seed 1234 (written by make_golden.py from the CPU oracle)\n")
        f.write(f"# in_scale={p['in_scale']} in_zp={p['in_zp']} out_scale={p['out_scale']} "
                f"out_zp={p['out_zp']}\n")
        for name, a in (("x", x), ("w", w), ("ws", ws), ("b", b), ("acc", acc), ("out", out)):
            _dump(f, name, a)


if __name__ == "__main__":
    linear_chain_8x64x32(os.path.join(HERE, "linear_chain_8x64x32.txt"))
    conv_t_small(os.path.join(HERE, "conv_t_1x3x5x4_k3s2p1op1.txt"))
