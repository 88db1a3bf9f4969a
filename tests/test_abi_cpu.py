"""CPU checks of the C ABI: the library loads, exports every declared entry
point, and validates shapes and sizes without touching a GPU."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[a-z ]+?\s(moe_\w+)\s*\(", src)))


def _lib():
    return pytest.importorskip("moe_layer_dsv3_gb300")


def test_header_declares_entry_points():
    names = _declared()
    for n in ("moe_route", "moe_schedule", "moe_dispatch", "moe_forward", "moe_backward", "moe_quantize_mxfp8",
              "moe_quantize_weights", "moe_workspace_size", "moe_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    m = _lib()
    for n in _declared():
        assert hasattr(m._lib, n), n
    assert sorted(m.exported_symbols()) == _declared()


def test_enums_match_header():
    m = _lib()
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    ws = re.findall(r"\bMOE_WS_(\w+)\b", src)
    seen = []
    for n in ws:
        if n not in seen:
            seen.append(n)
    assert seen[:-1] == m.WS_NAMES and seen[-1] == "COUNT"
    wq = []
    for n in re.findall(r"\bMOE_WQ_(\w+)\b", src):
        if n not in wq:
            wq.append(n)
    assert wq[:-1] == m.WQ_NAMES and wq[-1] == "COUNT"


def test_sizes_and_validation():
    m = _lib()
    cfg = m.config(256, 256, 8, 2, 1, 1, 128, 0)
    ws = m.moe_workspace_size(cfg)
    wq = m.moe_weights_size(cfg)
    # weights: 4 orientations of 3*d*I fp8 values per expert plus 1/32 scales
    assert wq >= 8 * (2 * 3 * 256 * 128) * 33 // 32
    assert ws > 256 * 2 * 256 * 2          # at least the per-assignment outputs
    big = m.config(16384, 7168, 256, 8, 8, 4, 2048, 1, 640)
    assert m.moe_workspace_size(big) > m.moe_workspace_size(m.config(4096, 7168, 256, 8, 8, 4, 2048, 1, 640))
    for bad in (m.config(256, 200, 8, 2), m.config(256, 256, 8, 9), m.config(256, 256, 8, 2, 3, 1),
                m.config(256, 256, 8, 2, 1, 1, 100), m.config(256, 256, 8, 2, 1, 1, 128, 2),
                m.config(256, 256, 8, 2, 1, 1, 128, 0, 100), m.config(256, 256, 8, 2, 8, 1)):
        with pytest.raises(m.MoeError):
            m.moe_workspace_size(bad)


def test_views_are_disjoint_and_inside_workspace():
    m = _lib()
    cfg = m.config(300, 256, 16, 4, 4, 2, 256, 1, 128)
    total = m.moe_workspace_size(cfg)
    spans = []
    for name in m.WS_NAMES:
        p, n = m.moe_ws_view(cfg, 1 << 20, name)
        off = p - (1 << 20)
        assert off % 256 == 0 and off + n <= total
        spans.append((off, off + n))
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0


def test_misaligned_buffers_are_rejected_before_any_launch():
    # Argument checks run before the device check, so on a host without a GPU a
    # misaligned buffer gives MOE_ERR_INVALID_ARG and an aligned one gets as
    # far as MOE_ERR_UNSUPPORTED_ARCH; nothing is launched or dereferenced.
    m = _lib()
    cfg = m.config(256, 256, 8, 2, 1, 1, 128, 1)
    A, B = 1 << 20, (1 << 20) + 8           # 16-byte aligned and misaligned fake device addresses

    def rc(call):
        try:
            call()
            return m.MOE_OK
        except m.MoeError as e:
            return e.code

    calls = {
        "forward": lambda x: m.moe_forward(cfg, x, A, A, A, A),
        "backward": lambda x: m.moe_backward(cfg, A, A, A, A, x, A, A, A, A, A, A, A, A),
        "route": lambda x: m.moe_route(cfg, x, A, A, A, A, A),
        "dispatch": lambda x: m.moe_dispatch(cfg, A, x),
        "quantize_weights": lambda x: m.moe_quantize_weights(cfg, A, x, A, A, A),
    }
    for name, call in calls.items():
        assert rc(lambda: call(B)) == m.MOE_ERR_INVALID_ARG, name
        assert rc(lambda: call(A)) != m.MOE_ERR_INVALID_ARG, name
