"""SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based generator: draw(key, c) is
the c-th output (0-based) of the SplitMix64 sequence seeded with `key`.
Host-side small draws (weights, masks, permutations) live here; the element
values are drawn by the same definition in synth.c and synth_dev.cu."""

MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def mix(z: int) -> int:
    z &= MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def draw(key: int, c: int) -> int:
    return mix(key + (c + 1) * GAMMA)


def stream(seed: int, tag: int) -> int:
    """Key of an independent stream: output `tag` of the sequence seeded with `seed`."""
    return draw(seed, tag)


def below(seed: int, tag: int, n: int) -> int:
    """Uniform integer in [0, n) (multiply-shift on the top 32 bits)."""
    u = draw(stream(seed, tag), 0) >> 32
    return (u * n) >> 32


def unit(seed: int, tag: int) -> float:
    """Uniform double in [0, 1) from the top 53 bits."""
    return (draw(stream(seed, tag), 0) >> 11) * (1.0 / (1 << 53))


def permutation(seed: int, tag: int, n: int) -> list:
    """Fisher-Yates shuffle of 0..n-1 driven by the stream (seed, tag)."""
    key = stream(seed, tag)
    a = list(range(n))
    for i in range(n - 1, 0, -1):
        j = ((draw(key, i) >> 32) * (i + 1)) >> 32
        a[i], a[j] = a[j], a[i]
    return a
