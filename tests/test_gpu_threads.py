"""Several host threads calling w4a16_gemm at once, on their own streams, from the first call on.

The library keeps per-device state that the first calls fill in: the error word, SM counts, the
kernels' shared-memory opt-ins and pads, the cluster capacities and the tensor maps of x.  A fresh
process starts four threads that call it at once for decode (1 and 8 rows), mid-size (24 rows) and
tensor-core (129 and 512 rows) shapes of fp16 and bf16 layers; every result must equal, bit for bit,
the one the same process computes afterwards from a single thread (each path adds in a fixed
order), and the error word must stay clean.
"""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r'''
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    import numpy as np
    import torch
    import w4a16_group_wise_gb300 as w4
    from w4a16_group_wise_gb300 import inputs

    dev = torch.device("cuda", 0)
    cases = [("qkv", 1, "f16"), ("gate_up", 8, "f16"), ("down", 24, "f16"), ("qkv", 129, "f16"),
             ("gate_up", 512, "f16"), ("down", 512, "f16"), ("qkv", 24, "bf16"), ("down", 512, "bf16")]
    layers = {}
    for name, M, dt in cases:
        K, N = inputs.SHAPES[name]
        h = inputs.make_weights(K, N, 128, seed=K + N)
        sc = torch.from_numpy(h["scales"]).to(dev)
        if dt == "bf16":
            sc = sc.float().to(torch.bfloat16)
        t = [torch.from_numpy(h["qweight"]).to(dev), torch.from_numpy(h["qzeros"]).to(dev), sc]
        packed = w4.repack(*t, K, N, 128)
        x = torch.from_numpy(inputs.make_x(M, K, seed=M)).to(dev)
        if dt == "bf16":
            x = x.float().to(torch.bfloat16)
        layers[(name, M, dt)] = (packed, x, K, N)
    torch.cuda.synchronize()

    results = {}
    errors = []
    start = threading.Barrier(4)

    def work(tid):
        try:
            s = torch.cuda.Stream(device=dev)
            start.wait()
            with torch.cuda.stream(s):
                for rep in range(3):
                    for i, key in enumerate(cases):
                        if (i + tid) % 2:
                            continue
                        packed, x, K, N = layers[key]
                        y = w4.gemm(x, packed, key[1], N, K, 128, stream=s)  # a workspace per stream
                        results[(tid, rep, key)] = y
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert w4.last_device_error() == 0
    for key in cases:
        packed, x, K, N = layers[key]
        ref = w4.gemm(x, packed, key[1], N, K, 128)
        torch.cuda.synchronize()
        for (tid, rep, k2), y in results.items():
            if k2 == key:
                assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (tid, rep, key)
    assert w4.last_device_error() == 0
    print("ok", len(results))
''')


@pytest.mark.gpu
def test_concurrent_first_calls_from_host_threads():
    env = dict(os.environ)
    proc = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=600,
                          cwd=ROOT, env=env)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-4000:]
    assert proc.stdout.strip().startswith("ok"), proc.stdout[-2000:]


SCRIPT_WS = textwrap.dedent(r'''
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    import torch
    import w4a16_group_wise_gb300 as w4
    from w4a16_group_wise_gb300 import binding, inputs

    # every split-K launch through the workspace: the binding's default workspace is per stream
    w4.set_option(binding.OPT_SPLITK_REDUCTION, binding.SPLITK_GLOBAL)
    dev = torch.device("cuda", 0)
    cases = [("down", 512), ("qkv", 129), ("square", 40)]
    layers = {}
    for name, M in cases:
        K, N = inputs.SHAPES[name]
        assert w4.workspace_bytes(M, N, K, 128) > 0, name
        h = inputs.make_weights(K, N, 128, seed=K + M)
        t = [torch.from_numpy(h[k]).to(dev) for k in ("qweight", "qzeros", "scales")]
        layers[(name, M)] = (w4.repack(*t, K, N, 128), torch.from_numpy(inputs.make_x(M, K, seed=M)).to(dev), K, N)
    torch.cuda.synchronize()
    results, errors = {}, []
    start = threading.Barrier(3)

    def work(tid):
        try:
            s = torch.cuda.Stream(device=dev)
            start.wait()
            with torch.cuda.stream(s):
                for rep in range(4):
                    for key in cases:
                        packed, x, K, N = layers[key]
                        results[(tid, rep, key)] = w4.gemm(x, packed, key[1], N, K, 128, stream=s)
            s.synchronize()
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert w4.last_device_error() == 0
    for key in cases:
        packed, x, K, N = layers[key]
        ref = w4.gemm(x, packed, key[1], N, K, 128)
        torch.cuda.synchronize()
        for (tid, rep, k2), y in results.items():
            if k2 == key:
                assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (tid, rep, key)
    print("ok", len(results))
''')


@pytest.mark.gpu
def test_concurrent_streams_get_their_own_default_workspace():
    """Three host threads on three streams run split-K problems through the workspace reduction at
    once; the binding's default workspace is per stream, so their arrival counters and partial
    tiles never mix: every result equals the single-threaded one bit for bit."""
    proc = subprocess.run([sys.executable, "-c", SCRIPT_WS, ROOT], capture_output=True, text=True, timeout=600,
                          cwd=ROOT, env=dict(os.environ))
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-4000:]
    assert proc.stdout.strip().startswith("ok"), proc.stdout[-2000:]
