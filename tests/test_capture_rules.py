"""Static checks of the library sources for the stream-capture contract the
header states: every call except lsm_get_device_status issues only kernel
launches and asynchronous memsets on the caller's stream, so that it can be
captured into a CUDA graph. A synchronizing, allocating or synchronous-copy
CUDA runtime call anywhere else would break capture (or stall the stream)."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "lsm_replacement_merge_gb300", "csrc")

# calls that synchronize, allocate or copy synchronously
FORBIDDEN = re.compile(
    r"\b(cudaMalloc\w*|cudaFree\w*|cudaDeviceSynchronize|cudaStreamSynchronize|"
    r"cudaEventSynchronize|cudaMemcpy|cudaMemcpyToSymbol|cudaMemcpyFromSymbol|cudaMemset|"
    r"cudaHostAlloc|cudaMallocHost|cudaDeviceReset)\s*\(")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name)) as f:
                yield name, f.read()


def _strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def _function_spans(text, name):
    """[start, end) of the body of every definition of function `name`."""
    spans = []
    for m in re.finditer(r"\b%s\s*\([^;{]*\)\s*\{" % re.escape(name), text):
        depth, i = 1, m.end()
        while depth and i < len(text):
            depth += {"{": 1, "}": -1}.get(text[i], 0)
            i += 1
        spans.append((m.start(), i))
    return spans


def test_sources_found():
    names = [n for n, _ in _sources()]
    assert "api.cu" in names and "replacement.cu" in names and "fc.cu" in names


def test_no_synchronous_calls_outside_the_status_read():
    bad = []
    for name, text in _sources():
        code = _strip_comments(text)
        allowed = _function_spans(code, "lsm_get_device_status") if name == "api.cu" else []
        for m in FORBIDDEN.finditer(code):
            if any(a <= m.start() < b for a, b in allowed):
                continue
            line = code.count("\n", 0, m.start()) + 1
            bad.append("%s:%d %s" % (name, line, m.group(1)))
    assert not bad, "calls that break stream capture: " + ", ".join(bad)


def test_the_status_read_is_the_one_synchronizing_call():
    code = _strip_comments(dict(_sources())["api.cu"])
    spans = _function_spans(code, "lsm_get_device_status")
    assert len(spans) == 1
    body = code[spans[0][0]:spans[0][1]]
    assert "cudaStreamSynchronize" in body


def test_the_checker_sees_a_planted_call():
    # the pattern and the comment stripping catch a call in code, not in a comment
    planted = "void f() {\n  // cudaMalloc(&p, 4);\n  cudaMalloc(&p, 4);\n}\n"
    code = _strip_comments(planted)
    hits = [m.group(1) for m in FORBIDDEN.finditer(code)]
    assert hits == ["cudaMalloc"]
    assert not list(FORBIDDEN.finditer(_strip_comments("// cudaMemset(x, 0, 4);\n")))
    assert not list(FORBIDDEN.finditer("cudaMemsetAsync(x, 0, 4, s);"))
