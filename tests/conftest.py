import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Parity margins that tests record with record_property('parity', {...}); printed in a
# short block at the end of the run so that they survive a quiet (-q) run's output.
_PARITY = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_runtest_logreport(report):
    if report.when == 'call':
        for key, value in report.user_properties:
            if key == 'parity':
                _PARITY.append(value)


def pytest_terminal_summary(terminalreporter):
    if not _PARITY:
        return
    terminalreporter.write_line('parity margins (worst relative error / tolerance):')
    for p in _PARITY:
        errs = ', '.join(f'{k} {v:.2e}' for k, v in p.items()
                         if k not in ('case', 'tol', 'heads', 'steps') and isinstance(v, float))
        terminalreporter.write_line(f"  {p['case']}: {errs} (tol {p['tol']:.0e}, "
                                    f"{p.get('heads', '?')} heads x {p.get('steps', '?')} steps)")
