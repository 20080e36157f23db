import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


def pytest_terminal_summary(terminalreporter):
    """Report the 2x-naive gate: how close each gated tensor came to its bound
    (err / floor; the bound is 2) and every use of the pages' 1e-3 slack."""
    try:
        from parity import GATE_LOG
    except ImportError:
        return
    if not GATE_LOG:
        return
    tr = terminalreporter
    tr.section("2x-naive gate report (err / floor; bound 2)")
    by = {}
    for e in GATE_LOG:
        by.setdefault(e["name"], []).append(e)
    for name in sorted(by):
        rs = [e["ratio"] for e in by[name] if e["floor"] > 0]
        if rs:
            tr.write_line(f"{name:>3}: {len(by[name])} gates, err/floor min {min(rs):.2f} "
                          f"median {sorted(rs)[len(rs) // 2]:.2f} max {max(rs):.2f}")
    worst = sorted(GATE_LOG, key=lambda e: -e["ratio"] if e["floor"] > 0 else 0)[:5]
    for e in worst:
        tr.write_line(f"  highest: {e['test']} {e['name']} err {e['err']:.3e} floor "
                      f"{e['floor']:.3e} ratio {e['ratio']:.2f}")
    slack = [e for e in GATE_LOG if e["slack"]]
    tr.write_line(f"slack (2 x floor + 1e-3, floor < 1e-4) used {len(slack)} times" +
                  (":" if slack else ""))
    for e in slack:
        tr.write_line(f"  {e['test']} {e['name']} err {e['err']:.3e} floor {e['floor']:.3e}")
