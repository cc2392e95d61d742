"""Write angle_table.inc: sin and cos of j * pi / 256, j = 0..72, as float-float.

Each entry is (fl32(sin x), fl32(sin x - fl32(sin x)), fl32(cos x),
fl32(cos x - fl32(cos x))) for x = j * pi / 256, evaluated with 160-bit
mpmath arithmetic; the second step of the argument reduction in storage.cuh
looks them up.  Also prints the float split of the step pi / 256 and 256 / pi.
Run: python gen_angle_table.py  (needs mpmath; the output is committed)
"""
import math
import os

import mpmath as mp
import numpy as np

mp.mp.prec = 160
N = 73


def fl(x) -> np.float32:
    return np.float32(float(x))


def main():
    step = mp.pi / 256
    lines = ["// sin(j pi / 256), cos(j pi / 256) for j = 0..72 as float-float",
             "// {sin hi, sin lo, cos hi, cos lo}; written by gen_angle_table.py",
             f"__device__ const float4 kSinCosStep[{N}] = {{"]
    for j in range(N):
        s, c = mp.sin(j * step), mp.cos(j * step)
        sh = fl(s)
        sl = fl(s - mp.mpf(float(sh)))
        ch = fl(c)
        cl = fl(c - mp.mpf(float(ch)))
        lines.append(f"    {{{float(sh).hex()}f, {float(sl).hex()}f, {float(ch).hex()}f, {float(cl).hex()}f}},")
    lines.append("};")
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "angle_table.inc")
    with open(out, "w") as f:
        f.write("\n".join(lines).replace("0x0.0p+0f", "0.0f") + "\n")
    m, e = math.frexp(float(step))
    hi = np.float32(math.ldexp(math.floor(m * 2 ** 17) / 2 ** 17, e))  # 17 significant bits
    lo = fl(step - mp.mpf(float(hi)))
    lo2 = fl(step - mp.mpf(float(hi)) - mp.mpf(float(lo)))
    print("step hi", float(hi).hex(), "lo", float(lo).hex(), "lo2", float(lo2).hex(),
          "256/pi", float(fl(256 / mp.pi)).hex())


if __name__ == "__main__":
    main()
