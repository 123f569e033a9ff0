"""The byte accounting behind the benchmark's GB/s and roofline figures, checked against the
figures the source pages print (tests/golden/page_figures.txt, one citation per line)."""
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def _rows():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, args, printed, tol, cite = (f.strip() for f in line.split("|", 4))
        kw = {k: float(v) if "." in v else int(v) for k, v in (a.split("=") for a in args.split())}
        rows.append((name, kw, float(printed.split()[0]), float(tol), cite))
    return rows


ROWS = _rows()


@pytest.mark.parametrize("name,kw,printed,tol,cite", ROWS, ids=[f"{r[0]}-{i}" for i, r in enumerate(ROWS)])
def test_page_figure(name, kw, printed, tol, cite):
    if name == "mamba_gbs":
        got = bench.mamba_page_bytes(kw["B"], kw["D"], kw["N"]) / (kw["us"] * 1e-6) / 1e9
    elif name == "mamba_pct":
        got = 100 * bench.mamba_page_bytes(kw["B"], kw["D"], kw["N"]) / (kw["us"] * 1e-6) / 600e9
    elif name == "mamba_vector_bytes":
        # the page's takeaway counts the five N-vectors only: B D 20 N bytes
        got = (bench.mamba_page_bytes(kw["B"], kw["D"], kw["N"]) - 24 * kw["B"] * kw["D"]) / 1e3
    elif name == "gemv_weight":
        got = bench.gemv_weight_bytes(kw["N"], kw["Kd"]) / 1e6
    elif name == "bf16_state_head":
        got = bench.state_tile_bytes(kw["V"], kw["K"], "bf16") / 1024
    elif name == "fused_layer":
        got = bench.fused_layer_bytes(kw["T"], kw["heads"], kw["D"]) / 1e9
    else:
        raise AssertionError(f"unknown figure {name}")
    assert abs(got - printed) <= tol, (name, kw, got, printed, cite)


def test_every_figure_is_cited():
    assert len(ROWS) >= 10
    for name, _, _, _, cite in ROWS:
        assert cite.startswith('"') and ", " in cite, name
