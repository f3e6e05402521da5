"""Linear layouts over F2 -- the oracle's own, plain implementation.

TEST INFRASTRUCTURE ONLY (tests/ and the smoke check import it; the product
path never does).  Independent of the C++ layout planner in the CUDA library.

Follows "A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs",
section "A Linear Layout Refresher":
  * "The Basic Idea": a layout maps hardware inputs (register, lane, warp, or a
    shared-memory offset) to output coordinates and is fixed by the images of
    the input bases 1, 2, 4, ...; the image of any index is the XOR of the
    images of the bases it decomposes into (a binary matrix on input bits).
  * "Dividing Layouts": L is divisible on the left by T when its matrix is
    block diagonal diag(T, R); the quotient is R.
and section "Lowering local_load to ds_load_tr in Triton":
  * cvt = dstLL.invertAndCompose(sharedLL) maps each destination hardware
    position to the shared offset that holds the same coordinates; sharedLL
    must be surjective for the lookup to succeed;
  * the same section's address computation inverts the full tile's shared
    layout (coordinates -> offset) before composing it with the repetition
    layout: ``invert`` below (bijective layouts with one input dimension).

Representation: ``ins`` is an ordered list of (input name, [basis images]);
each image is a tuple with one integer per output dimension.  ``outs`` is an
ordered list of (output name, size), sizes powers of two.
"""
from __future__ import annotations

from itertools import product
from typing import Dict, List, Sequence, Tuple

Image = Tuple[int, ...]


def _log2(n: int) -> int:
    if n < 1 or n & (n - 1):
        raise ValueError(f"{n} is not a power of two")
    return n.bit_length() - 1


class LinearLayout:
    def __init__(self, ins: Sequence[Tuple[str, Sequence[Sequence[int]]]],
                 outs: Sequence[Tuple[str, int]]):
        self.outs: List[Tuple[str, int]] = [(n, int(s)) for n, s in outs]
        for _, s in self.outs:
            _log2(s)
        nout = len(self.outs)
        self.ins: List[Tuple[str, List[Image]]] = []
        for name, bases in ins:
            imgs = []
            for b in bases:
                b = tuple(int(v) for v in b)
                if len(b) != nout:
                    raise ValueError(f"basis {b} of {name} has {len(b)} coords, want {nout}")
                imgs.append(b)
            self.ins.append((name, imgs))

    # -- basic queries -------------------------------------------------------
    def in_names(self) -> List[str]:
        return [n for n, _ in self.ins]

    def bases(self, name: str) -> List[Image]:
        for n, b in self.ins:
            if n == name:
                return b
        raise KeyError(name)

    def in_size(self, name: str) -> int:
        return 1 << len(self.bases(name))

    def out_size(self, name: str) -> int:
        return dict(self.outs)[name]

    def total_in_bits(self) -> int:
        return sum(len(b) for _, b in self.ins)

    def total_out_bits(self) -> int:
        return sum(_log2(s) for _, s in self.outs)

    # -- evaluation: XOR of the images of the set bits -----------------------
    def apply(self, **inputs: int) -> Image:
        acc = [0] * len(self.outs)
        for name, bases in self.ins:
            x = int(inputs.get(name, 0))
            if x >> len(bases):
                raise ValueError(f"{name}={x} out of range")
            for bit, img in enumerate(bases):
                if (x >> bit) & 1:
                    acc = [a ^ v for a, v in zip(acc, img)]
        return tuple(acc)

    # -- flattening to a bit matrix (columns = input bits, rows = output bits)
    def _flat_out(self, img: Image) -> int:
        v, shift = 0, 0
        for (_, size), c in zip(self.outs, img):
            v |= c << shift
            shift += _log2(size)
        return v

    def _unflat_out(self, v: int) -> Image:
        res, shift = [], 0
        for _, size in self.outs:
            w = _log2(size)
            res.append((v >> shift) & ((1 << w) - 1))
            shift += w
        return tuple(res)

    def columns(self) -> List[int]:
        return [self._flat_out(img) for _, bases in self.ins for img in bases]

    def rank(self) -> int:
        return _rank(self.columns())

    def is_surjective(self) -> bool:
        return self.rank() == self.total_out_bits()

    def is_injective(self) -> bool:
        return self.rank() == self.total_in_bits()

    def is_bijective(self) -> bool:
        return self.is_injective() and self.is_surjective()

    def invert(self, in_name: str = "offset") -> "LinearLayout":
        """Inverse of a bijective layout with a single input dimension.  The
        inverse's inputs are this layout's outputs, its single output is
        ``in_name``."""
        if len(self.ins) != 1 or not self.is_bijective():
            raise ValueError("invert needs a bijective layout with one input dim")
        cols = self.columns()
        n = len(cols)
        ins = []
        shift = 0
        for oname, size in self.outs:
            imgs = []
            for bit in range(_log2(size)):
                target = 1 << (shift + bit)
                sol = _solve(cols, target)
                imgs.append((sol,))
            ins.append((oname, imgs))
            shift += _log2(size)
        return LinearLayout(ins, [(self.ins[0][0] if in_name is None else in_name, 1 << n)])

    def invert_and_compose(self, shared: "LinearLayout") -> "LinearLayout":
        """cvt(x) = shared^{-1}(self(x)): for each input basis of ``self``, find
        the shared-layout input whose image is the same coordinate tuple."""
        if [o for o, _ in self.outs] != [o for o, _ in shared.outs]:
            raise ValueError("output dimensions differ")
        if not shared.is_surjective():
            raise ValueError("shared layout must be surjective")
        scols = shared.columns()
        sh_ins = shared.ins
        out_dims = [(name, 1 << len(bases)) for name, bases in sh_ins]
        res = []
        for name, bases in self.ins:
            imgs = []
            for img in bases:
                x = _solve(scols, self._flat_out(img))
                # split the solution bits over shared's input dims
                parts, shift = [], 0
                for _, sb in sh_ins:
                    w = len(sb)
                    parts.append((x >> shift) & ((1 << w) - 1))
                    shift += w
                imgs.append(tuple(parts))
            res.append((name, imgs))
        return LinearLayout(res, out_dims)

    def __eq__(self, other) -> bool:
        return isinstance(other, LinearLayout) and self.ins == other.ins and self.outs == other.outs

    def __repr__(self) -> str:
        return f"LinearLayout(ins={self.ins}, outs={self.outs})"


def identity_1d(size: int, in_name: str, out_name: str) -> LinearLayout:
    return LinearLayout([(in_name, [(1 << i,) for i in range(_log2(size))])], [(out_name, size)])


def divide_left(L: LinearLayout, T: LinearLayout):
    """Block-diagonal factorisation L = diag(T, R); returns R or None.

    T's input bases must be the first bases of the same-named input dims of L,
    with identical images; every other basis of L must be zero on the output
    bits that T covers (the low bits of T's output dims); R keeps those other
    bases with T's output bits shifted away."""
    t_in = dict((n, b) for n, b in T.ins)
    t_out = dict(T.outs)
    out_names = [n for n, _ in L.outs]
    for n in t_out:
        if n not in out_names:
            return None
    low = [(_log2(t_out[n]) if n in t_out else 0) for n in out_names]
    t_pos = [out_names.index(n) for n, _ in T.outs]
    rest = []
    for name, bases in L.ins:
        tb = t_in.get(name, [])
        if len(tb) > len(bases):
            return None
        for i, img in enumerate(tb):
            want = [0] * len(out_names)
            for j, p in enumerate(t_pos):
                want[p] = img[j]
            if tuple(bases[i]) != tuple(want):
                return None
        kept = []
        for img in bases[len(tb):]:
            if any(c & ((1 << w) - 1) for c, w in zip(img, low)):
                return None
            kept.append(tuple(c >> w for c, w in zip(img, low)))
        rest.append((name, kept))
    outs = [(n, s >> lw) for (n, s), lw in zip(L.outs, low)]
    return LinearLayout(rest, outs)


def _rank(cols: List[int]) -> int:
    basis: Dict[int, int] = {}
    for c in cols:
        v = c
        while v:
            h = v.bit_length() - 1
            if h in basis:
                v ^= basis[h]
            else:
                basis[h] = v
                break
    return len(basis)


def _solve(cols: List[int], target: int) -> int:
    """Find x (bitmask over columns) with XOR_{i in x} cols[i] == target."""
    # Gaussian elimination carrying the combination masks.
    rows: Dict[int, Tuple[int, int]] = {}
    for i, c in enumerate(cols):
        v, m = c, 1 << i
        while v:
            h = v.bit_length() - 1
            if h in rows:
                rv, rm = rows[h]
                v ^= rv
                m ^= rm
            else:
                rows[h] = (v, m)
                break
    v, m = target, 0
    while v:
        h = v.bit_length() - 1
        if h not in rows:
            raise ValueError("target not in the span")
        rv, rm = rows[h]
        v ^= rv
        m ^= rm
    return m


def enumerate_map(L: LinearLayout):
    """All (inputs, image) pairs, inputs as a dict -- brute force helper."""
    names = L.in_names()
    ranges = [range(L.in_size(n)) for n in names]
    for vals in product(*ranges):
        d = dict(zip(names, vals))
        yield d, L.apply(**d)
