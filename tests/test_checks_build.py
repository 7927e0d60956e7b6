"""The bounds-checked build (-DMLA_CHECKS): every kernel of the library, its
copies, shared-memory exchanges and output stores checked against the sizes
they must stay within (the memory checker is not available here, so the
library checks itself).  A failed check would raise MLA_DEVERR_CHECK with the
site's bit and skip the access.  The build goes to a temporary directory and
runs in a child process (the binding loads one library per process); each
case must raise no device flag and meet the oracle."""

import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys
    sys.path.insert(0, sys.argv[1])
    import numpy as np, torch
    from mla_query_projection_gb300 import binding as B
    from mla_query_projection_gb300 import synthetic as S
    from mla_query_projection_gb300.runner import DecodeStep
    from tests.parity_util import check_against_oracle
    B.load(sys.argv[2])
    torch.cuda.set_device(0)
    cases = [
        # (batch, heads, layout, path): every kernel the dispatch reaches
        (1, 64, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),        # paired, 8 tokens
        (12, 128, S.LAYOUT_DS_MLA, B.MLA_PATH_AUTO),    # paired, 16 tokens
        (40, 64, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),       # wide, single-head rope units
        (64, 127, S.LAYOUT_DS_MLA, B.MLA_PATH_AUTO),    # wide, two-head rope units
        (70, 16, S.LAYOUT_NVFP4_DS_MLA, B.MLA_PATH_AUTO),  # wide, two slices
        (3, 16, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),        # partials kernel
        (1, 64, S.LAYOUT_E4M3, B.MLA_PATH_FMA),         # small-batch FMA, pairs
        (2, 16, S.LAYOUT_DS_MLA, B.MLA_PATH_FMA),       # small-batch FMA, larger clusters
        (7, 128, S.LAYOUT_E4M3, B.MLA_PATH_FMA),        # small-batch FMA, 8 tokens a CTA
    ]
    for batch, heads, layout, path in cases:
        inp = S.make_inputs(batch=batch, heads=heads, layout=layout, pages=16, seed=3000 + batch + heads)
        st = DecodeStep(inp)
        assert st.set_path(path) == B.MLA_OK
        assert st.decode() == B.MLA_OK
        out = st.results()
        flags = st.error_flags()
        st.close()
        assert flags == 0, (batch, heads, path, hex(flags))
        check_against_oracle(out, inp)
        print("ok", batch, heads, path, flush=True)
    # the hand-off kernel (allocation-free entry point)
    inp = S.make_inputs(batch=20, heads=32, layout=S.LAYOUT_E4M3, pages=16, seed=3100)
    st = DecodeStep(inp)
    flags = torch.zeros(1, dtype=torch.int32, device=st.q_a.device)
    assert B.mla_query_decode_noalloc(
        st.heads, st.w_qb, st.w_uk, st.gamma_q, st.gamma_kv, st.eps, st.batch, st.q_a,
        st.strides[0], st.kv_c, st.strides[1], st.k_pe, st.strides[2], st.slots, st.cache,
        st.num_pages, st.page_size, st.layout, st.k_scale, st.q_latent, st.q_pe, st.q_c, flags,
        torch.cuda.current_stream()) == B.MLA_OK
    out = st.results()
    assert int(flags.item()) == 0, hex(int(flags.item()))
    check_against_oracle(out, inp)
    st.close()
    print("ok noalloc", flush=True)
""")


def test_checks_build_every_kernel(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_query_projection_gb300 import build

    lib = build.build(out_dir=str(tmp_path / "checks"), extra=("-DMLA_CHECKS",))
    p = subprocess.run([sys.executable, "-c", CHILD, ROOT, lib], capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout[-3000:] + p.stderr[-3000:]
    assert p.stdout.count("ok") == 10, p.stdout
