"""Layer-structure arithmetic of the X-MoD stack (test infrastructure).

Sources: "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
Mixture-of-Depths" reading notes --
  Eq. 1   MoD stack ([Sparse(K)] + [Dense]) x N
  Eq. 2   MoD total/active ratio 2K/(K+1)
  Eq. 3   X-MoD stack [Dense] x N0 + ([Sparse(K)] x AK + [Dense]) x N1
  Eq. 4   total parameters N = N_layer (N0 + N1 (1 + AK))
  Eq. 5   active-equivalent parameters N_act = N_layer (N0 + N1 (1 + A))
  Eq. 34-36, Table 6, Table 9: the concrete stacks and their sizes;
  "mechanism controls", Table 2 / Table 7: the Routed-FFN variant, where each group of
  K routed layers keeps its FFN only and one full-sequence attention module serves the
  group: ([FullAttn] + [Routed-FFN] x K) x A between the dense anchors.
"""
from fractions import Fraction

DENSE, SPARSE, ATTN, RFFN = 0, 1, 2, 3


def _ak(A, K) -> int:
    ak = Fraction(A) * K
    if ak.denominator != 1 or ak < 1:
        raise ValueError(f"A*K must be a positive integer, got A={A}, K={K}")
    return int(ak)


def schedule(N0: int, N1: int, A, K: int) -> list:
    """Eq. 3: layer kinds in execution order. MoD (Eq. 1) is N0=0, A=1/K."""
    ak = _ak(A, K)
    return [DENSE] * N0 + ([SPARSE] * ak + [DENSE]) * N1


def schedule_segments(N0: int, segments) -> list:
    """Heterogeneous variant (Eq. 35): dense prefix, then (AK, repeats) segments,
    each segment being ([Sparse] x AK + [Dense]) x repeats."""
    kinds = [DENSE] * N0
    for ak, reps in segments:
        kinds += ([SPARSE] * int(ak) + [DENSE]) * int(reps)
    return kinds


def schedule_routed_ffn(N0: int, segments, K: int) -> list:
    """The Routed-FFN counterpart of schedule_segments: every segment (AK, repeats)
    becomes (([FullAttn] + [Routed-FFN] x K) x A + [Dense]) x repeats, A = AK / K."""
    kinds = [DENSE] * N0
    for ak, reps in segments:
        A, rem = divmod(int(ak), K)
        if rem:
            raise ValueError("a Routed-FFN segment needs AK divisible by K")
        kinds += (([ATTN] + [RFFN] * K) * A + [DENSE]) * int(reps)
    return kinds


def attention_modules(kinds) -> int:
    """Full-sequence attention modules: the dense anchors' and the FullAttn layers'."""
    return sum(1 for k in kinds if k in (DENSE, ATTN))


def ffn_depth(kinds) -> int:
    """Depth counted by FFN layers (Table 7 counts the Routed-FFN variants this way)."""
    return sum(1 for k in kinds if k in (DENSE, SPARSE, RFFN))


def physical_layers(kinds) -> int:
    return len(kinds)


def active_layers(kinds, K: int) -> Fraction:
    """Layers a token passes on average: a dense layer counts 1, a sparse layer 1/K."""
    n_dense = sum(1 for k in kinds if k == DENSE)
    n_sparse = sum(1 for k in kinds if k == SPARSE)
    return Fraction(n_dense) + Fraction(n_sparse, K)


def total_over_active(kinds, K: int) -> Fraction:
    return Fraction(physical_layers(kinds)) / active_layers(kinds, K)


def eq2_mod_ratio(K: int) -> Fraction:
    """Eq. 2 closed form: 2 / (1 + 1/K) = 2K / (K + 1)."""
    return Fraction(2 * K, K + 1)


def eq4_total(N_layer, N0, N1, A, K):
    return N_layer * (N0 + N1 * (1 + _ak(A, K)))


def eq5_active(N_layer, N0, N1, A):
    return N_layer * (N0 + N1 * (1 + Fraction(A)))


def layer_params(d, hq, hkv, hd, F, router=False, kind=DENSE) -> int:
    """Parameters of one block as the oracle's block uses them: Wq, Wk, Wv, Wo,
    SwiGLU (gate, up, down), two RMSNorm gains, plus the router vector if asked.
    kind ATTN keeps the attention half (and its gain), RFFN the FFN half."""
    att = d * hq * hd + 2 * d * hkv * hd + hq * hd * d + d
    ffn = 3 * d * F + d
    p = att if kind == ATTN else ffn if kind == RFFN else att + ffn
    return p + (d if router else 0)


def model_params(kinds, d, hq, hkv, hd, F, vocab=0, tied=False, router=False) -> int:
    """Total parameters of a stack plus (un)tied input/output embeddings."""
    n = 0
    for k in kinds:
        n += layer_params(d, hq, hkv, hd, F, router=(router and k in (SPARSE, RFFN)), kind=k)
    n += (1 if tied else 2) * vocab * d
    return n
