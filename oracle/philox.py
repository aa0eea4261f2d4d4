"""Counter-based uniforms for speculative sampling (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The discussion thread "Support Eagle-3 Speculative Decoding in llama.cpp"
lists an acceptance / rejection (speculative sampling) strategy for the draft
tokens; the random numbers that strategy consumes are keyed here by
(seed, step, node, child) so that any verify step can be replayed exactly.

Generator: Philox4x32 with 10 rounds, written from its published definition
(Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC'11): a 4-word counter and a 2-word key; each round multiplies counter
words 0 and 2 by two fixed odd constants, forms the next counter from the
high/low product halves XORed with the other two words and the key, and the
key is advanced by two Weyl increments between rounds.

Mapping used by both the oracle and the library (written independently on
each side):
    key     = (seed & 0xffffffff, seed >> 32)
    counter = (step & 0xffffffff, step >> 32, node, child)
    u       = (first output word >> 8) * 2**-24          (exact in fp32/fp64)
The residual (bonus) draw at a node uses child = 0xffffffff.
"""

_MASK32 = 0xFFFFFFFF
# Multipliers and Weyl key increments of Philox4x32 (SC'11, Table/Sec. on
# Philox-4x32): odd multipliers and the golden-ratio / sqrt(3)-1 increments.
_MUL_A = 0xD2511F53
_MUL_B = 0xCD9E8D57
_WEYL_A = 0x9E3779B9
_WEYL_B = 0xBB67AE85

RESIDUAL_CHILD = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Ten Philox4x32 rounds on ``counter`` (4 ints) under ``key`` (2 ints)."""
    x0, x1, x2, x3 = (int(c) & _MASK32 for c in counter)
    k0, k1 = (int(k) & _MASK32 for k in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _WEYL_A) & _MASK32
            k1 = (k1 + _WEYL_B) & _MASK32
        prod_a = _MUL_A * x0          # multiplies counter word 0
        prod_b = _MUL_B * x2          # multiplies counter word 2
        hi_a, lo_a = prod_a >> 32, prod_a & _MASK32
        hi_b, lo_b = prod_b >> 32, prod_b & _MASK32
        x0, x1, x2, x3 = (hi_b ^ x1 ^ k0, lo_b, hi_a ^ x3 ^ k1, lo_a)
    return x0, x1, x2, x3


def uniform(seed, step, node, child):
    """u in [0, 1) with 24 random bits, keyed by (seed, step, node, child)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    word = philox4x32_10(
        (step & _MASK32, step >> 32, int(node) & _MASK32, int(child) & _MASK32),
        (seed & _MASK32, seed >> 32),
    )[0]
    return (word >> 8) * (2.0 ** -24)
