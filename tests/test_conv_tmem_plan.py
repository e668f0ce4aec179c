"""Host-side check of the tensor-memory im2col conv kernel's index arithmetic.

The planner (csrc/api.cu, tconv_plan) sizes one raw input window per 64-value
K block; every producer lane then reads, for each K value of the block, the
window element at lane_off + table[k].  This test restates that arithmetic
and checks, for every tile, pixel and K value of many geometries, that

  * each offset lies inside the staged window (WB x HB x CB elements), so no
    shared-memory read leaves the window slot, and
  * the element it names is the input element the convolution needs: the
    window's (channel, row, column) maps back to x[n][ci][ih][iw] with
    ih = oh*sh - pt + r*dh and iw = ow*sw - pl + q*dw.

No GPU and no library call: the formulas are the ones the kernel and the
planner use, written out again here.
"""
import math

import pytest

WIN_MAX = 40960
TABLE_MAX = 3136


def plan(N, C, H, W, Co, kh, kw, st, pd, dl):
    sh, sw = st
    dh, dw = dl
    Ho = (H + pd[0] + pd[1] - dh * (kh - 1) - 1) // sh + 1
    Wo = (W + pd[2] + pd[3] - dw * (kw - 1) - 1) // sw + 1
    taps = kh * kw
    K = C * taps
    P = Ho * Wo
    if K % 8 or W % 8 or P <= 0:
        return None
    period = taps // math.gcd(64, taps)
    if period * 64 > TABLE_MAX:
        return None
    tiles_p = (P + 127) // 128
    nrows = 1
    for i in range(min(Wo // math.gcd(128, Wo), tiles_p)):
        s = (128 * i) % Wo
        nrows = max(nrows, (s + 127) // Wo + 1)
    nrows = min(nrows, Ho)
    lattice = sh > 1 and (kh == 1 or dh % sh == 0)
    HB = nrows + (kh - 1) * (dh // sh) if lattice else (nrows - 1) * sh + (kh - 1) * dh + 1
    esh = sh if lattice else 1
    x0 = -((pd[2] + 7) // 8) * 8
    xoff = -pd[2] - x0
    WB = (xoff + (Wo - 1) * sw + (kw - 1) * dw + 1 + 7) // 8 * 8
    CB = 64 // taps if 64 % taps == 0 else 63 // taps + 2
    raw = WB * HB * CB * 2
    if raw > WIN_MAX or WB > 256 or HB * esh > 256 or CB > 256:
        return None
    return dict(Ho=Ho, Wo=Wo, P=P, K=K, taps=taps, tiles_p=tiles_p, num_kb=(K + 63) // 64, period=period,
                HB=HB, WB=WB, CB=CB, esh=esh, x0=x0, xoff=xoff, rowmul=1 if lattice else sh,
                rstep=dh // sh if lattice else dh, sh=sh, sw=sw, dh=dh, dw=dw, pt=pd[0], pl=pd[2], kw=kw, C=C)


def table(p):
    tab = []
    plane = p["HB"] * p["WB"]
    for j in range(p["period"] * 64):
        ci, tap = divmod(j, p["taps"])
        r, q = divmod(tap, p["kw"])
        c_lo = ((j >> 6) << 6) // p["taps"]
        tab.append((ci - c_lo) * plane + r * p["rstep"] * p["WB"] + q * p["dw"])
    return tab


def check_geometry(geom):
    p = plan(*geom)
    assert p is not None, geom
    tab = table(p)
    size = p["WB"] * p["HB"] * p["CB"]
    Wo = p["Wo"]
    for pb in range(p["tiles_p"]):
        p0 = pb * 128
        oh_first = p0 // Wo
        y0 = oh_first * p["sh"] - p["pt"]
        for lane_px in range(128):
            px = min(p0 + lane_px, p["P"] - 1)
            oh, ow = divmod(px, Wo)
            lane_off = (oh - oh_first) * p["rowmul"] * p["WB"] + ow * p["sw"] + p["xoff"]
            for kb in range(p["num_kb"]):
                c_lo = (kb * 64) // p["taps"]
                trow = (kb % p["period"]) * 64
                for kl in range(64):
                    off = lane_off + tab[trow + kl]
                    assert 0 <= off < size, (geom, pb, lane_px, kb, kl, off, size)
                    k = kb * 64 + kl
                    ci, tap = divmod(k, p["taps"])
                    r, q = divmod(tap, p["kw"])
                    wc, rem = divmod(off, p["HB"] * p["WB"])
                    wr, wx = divmod(rem, p["WB"])
                    # window element -> input coordinates
                    assert c_lo + wc == ci, (geom, k)
                    assert y0 + wr * p["esh"] == oh * p["sh"] - p["pt"] + r * p["dh"], (geom, k)
                    assert p["x0"] + wx == ow * p["sw"] - p["pl"] + q * p["dw"], (geom, k)
    return p


GEOMETRIES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation)
    (8, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)),       # 3x3 s1 workload
    (16, 128, 64, 64, 256, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2)),     # 3x3 s2 d2 workload
    (16, 128, 64, 64, 256, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1)),     # 1x1 s2 workload
    (1, 16, 16, 16, 24, 3, 3, (2, 2), (1, 1, 1, 1), (1, 1)),        # s2 d1: no row lattice
    (2, 8, 40, 200, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)),        # Wo = 200 > 128
    (1, 16, 40, 8, 16, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)),         # Wo = 8: 16 rows per tile
    (1, 8, 20, 24, 16, 7, 7, (1, 1), (3, 3, 3, 3), (1, 1)),         # 49 taps
    (1, 24, 19, 48, 72, 3, 5, (1, 2), (0, 3, 2, 1), (2, 1)),        # asymmetric, mixed strides
    (2, 32, 24, 40, 48, 2, 2, (1, 1), (0, 1, 1, 0), (1, 1)),        # 2x2
    (1, 40, 13, 16, 40, 5, 5, (2, 1), (2, 2, 2, 2), (1, 1)),        # K = 1000 (tail)
    (1, 16, 7, 16, 16, 3, 3, (2, 1), (1, 1, 2, 2), (1, 2)),         # dh not a multiple of sh
    (1, 8, 30, 32, 8, 3, 3, (3, 3), (1, 1, 1, 1), (1, 1)),          # stride 3
]


@pytest.mark.parametrize("geom", GEOMETRIES, ids=lambda g: "x".join(map(str, g[:7])))
def test_window_offsets_in_bounds_and_correct(geom):
    p = check_geometry(geom)
    assert p["WB"] * p["HB"] * p["CB"] * 2 <= WIN_MAX


def test_workload_windows():
    # the planner takes the three conv workloads, with these windows
    p3 = plan(8, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1))
    p4 = plan(16, 128, 64, 64, 256, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2))
    p1 = plan(16, 128, 64, 64, 256, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1))
    assert (p3["WB"], p3["HB"], p3["CB"]) == (72, 6, 9)
    assert (p4["WB"], p4["HB"], p4["CB"], p4["esh"]) == (80, 6, 9, 2)
    assert (p1["WB"], p1["HB"], p1["CB"], p1["esh"]) == (64, 4, 64, 2)


def test_unsupported_geometries_fall_back():
    assert plan(1, 8, 16, 20, 8, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)) is None      # W % 8
    assert plan(1, 3, 16, 16, 8, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)) is None      # K = 27
    assert plan(1, 8, 64, 64, 8, 11, 11, (1, 1), (5, 5, 5, 5), (1, 1)) is None    # table too large
