"""CPU model of the window kernel's row ring (conv_window.cu).

The window kernel keeps each input row a tile needs in one slot of a ring per
phase of the vertical stride and lets consecutive tiles of a CTA reuse rows
already held.  This model restates the kernel's plan (tile shape, ring size,
slot of a row, what a tile writes) and checks, for every window test layer,
both MMA shapes and several grid sizes, that:
  * every slot an MMA operand reads holds the input row (image, segment, row)
    that operand needs when the MMA runs, for every stored output row;
  * the rows a tile writes never land in slots the previous tile's MMAs still
    read (unless the short ring makes that tile wait for those MMAs);
  * every slot index, mirror slot and operand run stays inside the ring.
A plausible mistake in the slot arithmetic (a wrong phase, a dropped mirror, a
base that moves by the wrong amount at an image boundary) fails one of these.
"""
import pytest

from deep_learning_convolution_gb300 import synth
from window_cases import WINDOW_CASES

WBM = 128
MAX_SMEM = 232448


def plan(layer, esz, pair):
    """The window kernel's tile and ring geometry (window_plan), or None."""
    C, H, W, K, R, S = layer.C, layer.H, layer.W, layer.K, layer.R, layer.S
    u, v, dh = layer.u, layer.v, layer.dil_h
    pt = layer.pad_top
    P = (H + layer.pad_top + layer.pad_bottom - (dh * (R - 1) + 1)) // u + 1
    Q = (W + layer.pad_left + layer.pad_right - (layer.dil_w * (S - 1) + 1)) // v + 1
    nb = v * C * esz
    if nb > 64:
        return None
    D = 16 if nb <= 16 else (32 if nb <= 32 else 64)
    A = -(-S // v)
    steps = (A * D + 31) // 32
    px_read = steps * 32 // D
    need = Q - 1 + px_read
    Qs = 32 if need <= 32 else (64 if need <= 64 else 128)
    J = WBM // Qs
    segs = 1 if J > 1 else -(-Q // WBM)
    PB = -(-P // J)
    span = 512 if D == 64 else 256
    if J > 1:
        slot_bytes = Qs * D
    else:
        step_px = 128 // D
        slot_px = -(-(WBM - 1 + px_read) // step_px) * step_px
        slot_bytes = -(-(slot_px * D) // span) * span
    rows = (J - 1) * u + (R - 1) * dh + 1
    kb_off = (-pt) // u
    kspan = (rows - 1 - pt) // u - kb_off + 1
    T = layer.N * PB * segs
    BN = -(-K // 16) * 16
    b_img = R * steps * (BN // 2 if pair else BN) * 32
    tail = -(-(px_read * D) // 1024) * 1024
    fixed = 1024 + -(-b_img // 1024) * 1024 + -(-(192 + 4 * rows + 8 * R * steps) // 16) * 16

    def ring_of(rs):
        return u * (rs + J - 1) * slot_bytes + tail

    RS, short = 2 * kspan, False
    if fixed + ring_of(RS) > MAX_SMEM:
        RS, short = kspan + J, True
    if fixed + ring_of(RS) > MAX_SMEM:
        return None
    return dict(P=P, J=J, segs=segs, PB=PB, rows=rows, kb_off=kb_off, kspan=kspan, RS=RS,
                RSJ=RS + J - 1, short=short, T=T, units=-(-T // 2) if pair else T, u=u,
                dh=dh, pt=pt, R=R)


def tile(p, t):
    rest = t // p["PB"]
    n = rest // p["segs"]
    return n, (rest - n * p["segs"]) * WBM, (t - rest * p["PB"]) * p["J"]


def slot_of(p, i, base):
    """Slot and ring position of tile row i (input row p0*u - pt + i)."""
    a = i - p["pt"]
    k = a // p["u"]
    assert 0 <= base < p["RS"] and 0 <= k - p["kb_off"] < p["kspan"]
    pos = base + k - p["kb_off"]
    if pos >= p["RS"]:
        pos -= p["RS"]
    return (a - k * p["u"]) * p["RSJ"] + pos, pos


def walk_cta(p, pair, ub, ue, rank, new_run_step=None):
    """Replays one CTA's units; new_run_step overrides the base step of a tile
    that starts a new run (kspan in the kernel)."""
    step = p["kspan"] if new_run_step is None else new_run_step
    ring = {}
    base = 0
    reads_prev = set()
    for uu in range(ub, ue):
        cont = not (uu == ub or uu % p["PB"] == 0)
        if pair and cont:
            t2 = uu + p["units"]
            cont = t2 >= p["T"] or t2 % p["PB"] != 0
        if uu > ub:
            base = (base + (p["J"] if cont else step)) % p["RS"]
        t = uu + p["units"] if (pair and rank) else uu
        writes = set()
        if t < p["T"]:
            n, q0, p0 = tile(p, t)
            i0 = max(0, p["rows"] - p["J"] * p["u"]) if cont else 0
            for i in range(i0, p["rows"]):
                h = p0 * p["u"] - p["pt"] + i
                s, pos = slot_of(p, i, base)
                assert 0 <= s < p["u"] * p["RSJ"]
                ring[s] = (n, q0, h)
                writes.add(s)
                if pos < p["J"] - 1:
                    m = s + p["RS"]
                    assert m // p["RSJ"] == s // p["RSJ"], "mirror slot left its phase"
                    ring[m] = (n, q0, h)
                    writes.add(m)
        if not (p["short"] and not cont):
            assert not writes & reads_prev, f"unit {uu} overwrote slots the previous MMAs read"
        reads = set()
        n, q0, p0 = tile(p, t) if t < p["T"] else (None, None, None)
        for r in range(p["R"]):
            s, pos = slot_of(p, r * p["dh"], base)
            assert pos + p["J"] - 1 < p["RSJ"], "operand run leaves the ring"
            reads.update(range(s, s + p["J"]))
            if t >= p["T"]:
                continue
            for j in range(p["J"]):
                if p0 + j >= p["P"]:
                    continue  # an output row that is not stored
                want = (n, q0, (p0 + j) * p["u"] + r * p["dh"] - p["pt"])
                assert ring.get(s + j) == want, f"unit {uu} filter row {r} output row {j}"
        reads_prev = reads


def short_ring(p):
    """The plan with the short ring (kspan + J slots per phase), which the
    kernel also takes to make room for staged rows."""
    q = dict(p)
    q["RS"] = min(p["RS"], p["kspan"] + p["J"])
    q["RSJ"] = q["RS"] + p["J"] - 1
    q["short"] = q["RS"] < 2 * p["kspan"] or p["short"]
    return q


@pytest.mark.parametrize("ring", ["planned", "short"])
@pytest.mark.parametrize("pair", [False, True], ids=["single", "pairs"])
@pytest.mark.parametrize("layer", WINDOW_CASES + [synth.WORKLOADS["alexnet"][0],
                                                  synth.WORKLOADS["overfeat"][0],
                                                  synth.WORKLOADS["speech"][0]],
                         ids=lambda l: l.name)
def test_ring_rows_reach_their_mmas(layer, pair, ring):
    esz = 4 if layer.dtype == "tf32" else 2
    p = plan(layer, esz, pair)
    assert p is not None, "the window kernel takes this layer"
    if ring == "short":
        p = short_ring(p)
    for grid in (152, 7, 1):
        G = min(grid, p["units"])
        for c in range(G):
            ub, ue = p["units"] * c // G, p["units"] * (c + 1) // G
            for rank in ((0, 1) if pair else (0,)):
                walk_cta(p, pair, ub, ue, rank)


def test_ring_model_catches_a_wrong_base_step():
    """A tile that starts a new image but moves the ring base by only J slots
    overwrites rows its predecessor's MMAs still read: the model must say so."""
    layer = WINDOW_CASES[0]
    p = plan(layer, 2, False)
    assert p["J"] < p["kspan"]
    with pytest.raises(AssertionError, match="overwrote"):
        for c in range(3):
            ub, ue = p["units"] * c // 3, p["units"] * (c + 1) // 3
            walk_cta(p, False, ub, ue, 0, new_run_step=p["J"])


def test_ring_random_layers():
    """Random few-channel layers (strides, dilation, pads, widths, batch): the
    plan, when it accepts the layer, keeps every operand on the right rows."""
    import numpy as np
    rng = np.random.default_rng(20260602)
    checked = 0
    for _ in range(300):
        u, v = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        R, S = int(rng.integers(1, 12)), int(rng.integers(1, 12))
        dh = int(rng.integers(1, 3))
        C = int(rng.integers(1, 9))
        pads = [int(rng.integers(0, 4)) for _ in range(4)]
        H = int(rng.integers(dh * (R - 1) + 1, 80))
        W = int(rng.integers(S, 300))
        n = int(rng.integers(1, 6))
        K = int(rng.choice([16, 32, 64, 96, 128]))
        layer = synth.Layer("rand", n, C, H, W, K, R, S, pad_top=pads[0], pad_bottom=pads[1],
                            pad_left=pads[2], pad_right=pads[3], u=u, v=v, dil_h=dh)
        for pair in (False, True):
            p = plan(layer, 2, pair)
            if p is None or p["P"] < 1:
                continue
            checked += 1
            for grid in (152, 5):
                G = min(grid, p["units"])
                for c in range(G):
                    ub, ue = p["units"] * c // G, p["units"] * (c + 1) // G
                    for rank in ((0, 1) if pair else (0,)):
                        walk_cta(p, pair, ub, ue, rank)
    assert checked > 100
