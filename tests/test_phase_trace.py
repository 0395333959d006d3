"""The phase-timeline report (CPU): stamps of a synthetic two-CTA, one-layer trace turn into
per-phase durations measured from the previous phase's last arrival."""
import numpy as np

from block_diffusion_drafter_forward_gb300 import phase_trace as pt


def test_table_from_synthetic_stamps(tmp_path):
    L, G, S = 1, 2, 10
    P = 2 + 6 * L
    t = np.zeros((G, P, S), dtype=np.uint64)
    base = 1_000_000
    for ph in range(P):
        for c in range(G):
            t[c, ph, 0] = base + ph * 10_000 + 1_000 + c * 100       # barrier passed
            t[c, ph, 7] = base + ph * 10_000 + 8_000 + c * 500       # arrival
    path = tmp_path / "trace.bin"
    with open(path, "wb") as fh:
        fh.write(np.array([G, P, S], dtype=np.int32).tobytes())
        fh.write(t.tobytes())
    back = pt.read_trace(str(path))
    assert back.shape == (G, P, S) and int(back[1, 3, 7]) == int(t[1, 3, 7])
    rows, total = pt.table(back, L)
    assert [r[0] for r in rows] == pt.phase_names(L)
    # phase 0 from the earliest stamp; later phases from the previous phase's last arrival
    assert abs(rows[0][1] - 7.5) < 1e-9
    for name, dur, cols in rows[1:]:
        assert abs(dur - 10.0) < 1e-9, name
        # barrier stamps 1.0 / 1.1 us into the phase, previous arrival 8.5 us into the last one
        assert abs(cols["barrier"][0] - 2.55) < 1e-9 and abs(cols["barrier"][1] - 2.6) < 1e-9
        assert cols["arrive"][1] == dur and "mma_last" not in cols
    assert abs(total - (7.5 + 10.0 * (P - 1))) < 1e-9


def test_table_reads_every_slot_the_trace_holds(tmp_path):
    """A trace with every slot reports the epilogue stamps too; an older, shorter trace
    reports the slots it holds and no others."""
    L, G = 1, 3
    P = 2 + 6 * L
    for S in (len(pt.SLOTS), 10):
        t = np.zeros((G, P, S), dtype=np.uint64)
        for ph in range(P):
            for c in range(G):
                for k in range(S):
                    t[c, ph, k] = 1_000_000 + ph * 10_000 + 100 * k + c
        path = tmp_path / f"trace{S}.bin"
        with open(path, "wb") as fh:
            fh.write(np.array([G, P, S], dtype=np.int32).tobytes())
            fh.write(t.tobytes())
        rows, _ = pt.table(pt.read_trace(str(path)), L)
        names = set(rows[3][2])
        assert names == set(pt.SLOTS[:S]), (S, names)
        # stamps 100 ns apart per slot: the slot's median sits 100 k ns after slot 0's
        r = rows[3][2]
        assert abs((r[pt.SLOTS[S - 1]][0] - r["barrier"][0]) - 0.1 * (S - 1)) < 1e-9
