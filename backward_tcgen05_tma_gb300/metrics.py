"""Work counts for the SwiGLU MLP used by the benchmark and the roofline.

FLOP convention of "[RFC] Full-pipeline SwiGLU MLP with forward/backward
co-optimization" (Liger-Kernel #1347), section "Training results": three
GEMMs of 2 M D H FLOPs each in forward (gate, up, down) and six in backward,
so forward = 6 M D H and forward + backward = 18 M D H, with M = B S.
"""


def fwd_flops(M: int, D: int, H: int) -> float:
    return 6.0 * M * D * H


def fwd_bwd_flops(M: int, D: int, H: int) -> float:
    return 18.0 * M * D * H


def nograd_intermediate_bytes(M: int, D: int, H: int, elt: int = 2) -> int:
    """Buffers the no-grad forward writes besides its inputs: A [M,H], Y [M,D]."""
    return (M * H + M * D) * elt


def nograd_algorithmic_bytes(M: int, D: int, H: int, elt: int = 2) -> int:
    """Bytes the no-grad forward must move at least once: the three weight
    matrices (3 D H), X read, A written then read back by the down
    projection, Y written."""
    return (3 * D * H + M * D + 2 * M * H + M * D) * elt


def fwd_bwd_algorithmic_bytes(M: int, D: int, H: int, elt: int = 2) -> int:
    """Bytes one forward + backward step moves at least once, kernel by kernel
    (each operand read once, each output written once per kernel):
      gate/up:   X, Wgu read; G, U, A written                M D + 2 H D + 3 M H
      down:      A, Wd read; Y written                      M H + D H + M D
      dG/dU:     dY, Wd, G, U read; dG, dU written          M D + D H + 4 M H
      dWd:       dY, A read; dWd written                    M D + M H + D H
      dWg/dWu:   dG, dU, X read; dWgu written               2 M H + M D + 2 H D
      dX:        dG, dU, Wgu read; dX written               2 M H + 2 H D + M D
    """
    md, mh, dh = M * D, M * H, D * H
    total = (md + 2 * dh + 3 * mh) + (mh + dh + md) + (md + dh + 4 * mh) + \
        (md + mh + dh) + (2 * mh + md + 2 * dh) + (2 * mh + 2 * dh + md)
    return total * elt
