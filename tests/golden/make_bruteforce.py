"""Write tests/golden/bruteforce_8x8x8.txt.

The pages print no worked example, so the fixture holds 8 x 8 x 8 closed-form
cases: inputs chosen so that the exact product, every partial sum and the
epilogue are representable in FP32 (identity, powers of two, small integers,
power-of-two alpha/beta).  For those inputs any correct FP32 GEMM -- and the
BF16x9 emulation in particular -- must return the exact result, which the
script takes from the oracle's FP64 reference and checks to be exact.

Run from the repository root:  python tests/golden/make_bruteforce.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def cases():
    r = np.random.Generator(np.random.PCG64(2024))
    out = []
    I = np.eye(8, dtype=np.float32)
    out.append(("identity_x_normal", I, r.standard_normal((8, 8)).astype(np.float32), 1.0, 0.0, None))
    out.append(("normal_x_identity", r.standard_normal((8, 8)).astype(np.float32), I, 1.0, 0.0, None))
    sg = lambda: np.where(r.random((8, 8)) < 0.5, -1.0, 1.0)  # noqa: E731
    out.append(("pow2", (sg() * np.ldexp(1.0, r.integers(-5, 6, (8, 8)))).astype(np.float32),
                (sg() * np.ldexp(1.0, r.integers(-5, 6, (8, 8)))).astype(np.float32), 1.0, 0.0, None))
    out.append(("int21_x_ternary", r.integers(-(1 << 20), 1 << 20, (8, 8)).astype(np.float32),
                r.integers(-1, 2, (8, 8)).astype(np.float32), 1.0, 0.0, None))
    out.append(("int13_x_int8_alpha2_betahalf", r.integers(-(1 << 11), 1 << 11, (8, 8)).astype(np.float32),
                r.integers(-(1 << 7), 1 << 7, (8, 8)).astype(np.float32), 2.0, -0.5,
                r.integers(-1000, 1000, (8, 8)).astype(np.float32)))
    out.append(("zeros_beta_quarter", np.zeros((8, 8), np.float32), r.standard_normal((8, 8)).astype(np.float32),
                1.0, 0.25, r.standard_normal((8, 8)).astype(np.float32)))
    return out


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bruteforce_8x8x8.txt")
    lines = ["# 8x8x8 closed-form GEMM cases, C = alpha*A*B + beta*C0, values as C99 hex floats.",
             "# Written by tests/golden/make_bruteforce.py from the oracle's FP64 reference;",
             "# every value here is exact in FP32, so any correct emulation returns C bitwise."]
    for name, A, B, alpha, beta, C0 in cases():
        if C0 is None:
            C0 = np.zeros((8, 8), np.float32)
        Cref, _ = oracle.gemm_ref(A, B, alpha=alpha, beta=beta, C0=C0)
        C = Cref.astype(np.float32)
        assert np.array_equal(C.astype(np.float64), Cref), name      # exact in FP32
        lines.append(f"case {name} {float(alpha).hex()} {float(beta).hex()}")
        for key, M in (("A", A), ("B", B), ("C0", C0), ("C", C)):
            lines.append(key)
            lines.extend(" ".join(float(v).hex() for v in row) for row in M)
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
