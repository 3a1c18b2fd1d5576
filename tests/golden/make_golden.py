"""Write oracle_digests.txt: SHA-256 digests of the CPU oracle's outputs on
small seeded cases.  Calls only the oracle and the seeded input generators.

The fixture pins the oracle build on one machine to the oracle build on another
(x86-64 here, aarch64 next to the GPU): both must produce the same bytes.

Run:  python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

CASES = [
    # name, M, N, K, kind, seed
    ("f32_m1_n256_k384", 1, 256, 384, 0, 11),
    ("f32_m3_n384_k256", 3, 384, 256, 0, 12),
    ("f32_m17_n128_k512", 17, 128, 512, 0, 13),
    ("ue8m0_m5_n256_k256", 5, 256, 256, 1, 14),
    ("ue8m0_m32_n128_k384", 32, 128, 384, 1, 15),
]


def digests(name, M, N, K, kind, seed):
    x = synth.x_bf16(M, K, seed=seed)
    w = synth.w_f32(N, K, seed=seed + 500)
    wq, ws = oracle.quant_weight_128x128(w, kind)
    y, xq, xs = oracle.linear(x, wq, ws, kind)
    out = {}
    for label, arr in (("x", x), ("wq", wq), ("ws", ws), ("xq", xq), ("xs", xs), ("y", y)):
        out[label] = hashlib.sha256(arr.tobytes()).hexdigest()[:32]
    return out


# RMSNorm producer cases (square root and division only: IEEE-exact on every
# machine).  name, M, K, kind, seed
RMS_CASES = [
    ("rms_f32_m3_k640", 3, 640, 0, 21),
    ("rms_ue8m0_m4_k1024", 4, 1024, 1, 22),
]


def rms_digests(name, M, K, kind, seed):
    x = synth.x_bf16(M, K, seed=seed)
    g = synth.gamma_bf16(K, seed=seed + 500)
    y, xq, xs = oracle.rmsnorm_quant(x, g, 1e-6, kind)
    return {label: hashlib.sha256(arr.tobytes()).hexdigest()[:32]
            for label, arr in (("x", x), ("gamma", g), ("y", y), ("xq", xq), ("xs", xs))}


def main():
    lines = ["# case label sha256[:32] -- written by make_golden.py from the oracle only"]
    for case in CASES:
        for label, h in digests(*case).items():
            lines.append(f"{case[0]} {label} {h}")
    for case in RMS_CASES:
        for label, h in rms_digests(*case).items():
            lines.append(f"{case[0]} {label} {h}")
    with open(os.path.join(HERE, "oracle_digests.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
