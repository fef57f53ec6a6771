"""Host-side checks of the C ABI; no GPU needed (nothing here launches)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def R():
    import __graft_entry__
    __graft_entry__.build()
    from linear_recurrent_sequence_gb300 import retention
    return retention


def declared_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if m.group(1) not in ("if", "sizeof"):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("retention_chunkwise_fwd", "retention_recurrent_step",
               "retention_parallel_fwd", "msr_layer_fwd"):
        assert op in names


def test_library_exports_every_declared_symbol(R):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(R.lib, n), f"{n} declared in include/ but not exported"
        assert n in R._SIGS, f"{n} has no binding"


def test_struct_layout_matches_header(R):
    # ret_desc: 6 ints, 2 enums, pointer, double, int, float, int64, int, 4 x int64[3]
    assert ctypes.sizeof(R.RetDesc) == 168
    assert R.RetDesc.sq.offset == 72
    assert ctypes.sizeof(R.MsrDesc) == 64


def _desc(R, **kw):
    g = (ctypes.c_double * 4)(0.9, 0.9, 0.9, 0.9)
    d = R.RetDesc()
    R.lib.retention_desc_init(ctypes.byref(d), 1, 2, 8, 4, 4, g)
    for k, v in kw.items():
        setattr(d, k, v)
    return d, g


def test_desc_init_defaults(R):
    d, _ = _desc(R)
    assert (d.chunk, d.in_dtype, d.out_dtype, d.rotate) == (64, 1, 1, 1)
    assert abs(d.theta_base - 10000.0) < 1e-12 and abs(d.gn_eps - 1e-6) < 1e-12
    assert list(d.sq) == [2 * 8 * 4, 8 * 4, 4]


@pytest.mark.parametrize("field,value", [
    ("B", -1), ("d_k", 3), ("d_k", 0), ("d_k", 512), ("d_v", 0), ("d_v", 2048),
    ("chunk", 0), ("chunk", 300), ("in_dtype", 7), ("norm_flags", 8), ("pos0", -1),
    ("pos0", 1 << 24), ("rotate", 2), ("theta_base", 0.0), ("H", 300)])
def test_invalid_descriptors_rejected(R, field, value):
    d, g = _desc(R, **{field: value})
    assert R.lib.retention_workspace_size(ctypes.byref(d)) == 0
    dummy = ctypes.c_void_p(256)
    st = R.lib.retention_chunkwise_fwd(ctypes.byref(d), dummy, dummy, dummy, None, None, None,
                                       None, dummy, dummy, 1 << 30, None)
    assert st == 1  # RET_EINVAL, before any launch


def test_gamma_out_of_range_rejected(R):
    g = (ctypes.c_double * 2)(0.9, 1.5)
    d = R.RetDesc()
    R.lib.retention_desc_init(ctypes.byref(d), 1, 2, 8, 4, 4, g)
    assert R.lib.retention_workspace_size(ctypes.byref(d)) == 0


def test_null_pointers_and_workspace(R):
    d, g = _desc(R)
    need = R.lib.retention_workspace_size(ctypes.byref(d))
    assert need >= 256
    dummy = ctypes.c_void_p(256)
    # null q
    assert R.lib.retention_chunkwise_fwd(ctypes.byref(d), None, dummy, dummy, None, None, None,
                                         None, dummy, dummy, need, None) == 1
    # workspace too small, missing, misaligned
    assert R.lib.retention_chunkwise_fwd(ctypes.byref(d), dummy, dummy, dummy, None, None, None,
                                         None, dummy, dummy, need - 1, None) == 3
    assert R.lib.retention_chunkwise_fwd(ctypes.byref(d), dummy, dummy, dummy, None, None, None,
                                         None, dummy, None, need, None) == 3
    assert R.lib.retention_chunkwise_fwd(ctypes.byref(d), dummy, dummy, dummy, None, None, None,
                                         None, dummy, ctypes.c_void_p(260), need, None) == 3


def test_recurrent_step_checks(R):
    d, g = _desc(R, N=1)
    dummy = ctypes.c_void_p(256)
    # N must be 1
    d2, g2 = _desc(R, N=2)
    assert R.lib.retention_recurrent_step(ctypes.byref(d2), dummy, dummy, dummy, dummy, None,
                                          dummy, dummy, 256, None) == 1
    # S must be 16-byte aligned
    assert R.lib.retention_recurrent_step(ctypes.byref(d), dummy, dummy, dummy,
                                          ctypes.c_void_p(260), None, dummy, dummy, 256,
                                          None) == 1
    # the third normalisation needs z
    d3, g3 = _desc(R, N=1, norm_flags=4)
    assert R.lib.retention_recurrent_step(ctypes.byref(d3), dummy, dummy, dummy, dummy, None,
                                          dummy, dummy, 256, None) == 1


def test_empty_batch_is_a_no_op(R):
    d, g = _desc(R, B=0)
    assert R.lib.retention_chunkwise_fwd(ctypes.byref(d), None, None, None, None, None, None,
                                         None, None, ctypes.c_void_p(256), 256, None) == 0


def test_status_strings(R):
    for code in range(6):
        assert R.lib.retention_status_string(code)
    assert R.lib.retention_last_cuda_error() == 0


def test_msr_workspace_and_checks(R):
    m, g = R.msr_desc(2, 4096, 2048, 8, 256, 512, [0.9] * 8, chunk=128)
    ws = R.lib.msr_workspace_size(ctypes.byref(m))
    assert ws >= 2 * 4096 * (2 * 8 * 256 + 3 * 8 * 512) * 2
    m2, g2 = R.msr_desc(2, 4096, 2048, 8, 3, 512, [0.9] * 8)  # odd d_k
    assert R.lib.msr_workspace_size(ctypes.byref(m2)) == 0


def test_backward_checks(R):
    dummy = ctypes.c_void_p(256)

    def bwd(d, dO=dummy, ws=dummy, nbytes=1 << 30):
        return R.lib.retention_chunkwise_bwd(ctypes.byref(d), dummy, dummy, dummy, None, dO,
                                             None, dummy, dummy, dummy, None, ws, nbytes, None)
    # GroupNorm on (the descriptor default) and the third normalisation are
    # not differentiated: RET_EUNSUPPORTED before any launch.
    d, g = _desc(R)
    assert bwd(d) == 2
    d, g = _desc(R, gn_eps=-1.0, norm_flags=4)
    assert bwd(d) == 2
    d, g = _desc(R, gn_eps=-1.0, norm_flags=3)
    need = R.lib.retention_backward_workspace_size(ctypes.byref(d))
    rows = 1 * 2 * 8 * 4 * 4  # B*H*N*d_k fp32 bytes
    assert need == 256 + 4 * ((rows + 255) // 256 * 256)
    assert bwd(d, dO=None) == 1
    assert bwd(d, nbytes=need - 1) == 3
    d, g = _desc(R, gn_eps=-1.0, d_k=3)
    assert R.lib.retention_backward_workspace_size(ctypes.byref(d)) == 0
    assert bwd(d) == 1
    d, g = _desc(R, gn_eps=-1.0, B=0)
    assert bwd(d, dO=None) == 0


def test_block_layout_workspace_and_checks(R):
    assert ctypes.sizeof(R.BlockDesc) == 72
    d, g = R.block_desc(2, 4096, 2048, 8, 256, 512, 4096, [0.9] * 8)
    m, g2 = R.msr_desc(2, 4096, 2048, 8, 256, 512, [0.9] * 8)
    need = R.lib.retnet_block_workspace_size(ctypes.byref(d))
    T = 2 * 4096
    assert need >= R.lib.msr_workspace_size(ctypes.byref(m)) + T * (2 * 2048 + 4096) * 2
    dummy = ctypes.c_void_p(256)
    args = [dummy] * 13
    # missing weight, small workspace, bad FFN width, bad LayerNorm epsilon
    bad = list(args)
    bad[11] = None
    assert R.lib.retnet_block_fwd(ctypes.byref(d), *bad, dummy, need, None) == 1
    assert R.lib.retnet_block_fwd(ctypes.byref(d), *args, dummy, need - 1, None) == 3
    d.d_ffn = 0
    assert R.lib.retnet_block_workspace_size(ctypes.byref(d)) == 0
    d.d_ffn, d.ln_eps = 4096, -1.0
    assert R.lib.retnet_block_fwd(ctypes.byref(d), *args, dummy, need, None) == 1
    d.ln_eps = 1e-5
    d.msr.B = 0
    assert R.lib.retnet_block_fwd(ctypes.byref(d), *([None] * 13), dummy, 1 << 30, None) == 0


def test_decode_stack_layout_and_checks(R):
    assert ctypes.sizeof(R.StackDesc) == 80 and ctypes.sizeof(R.LayerWeights) == 88
    d, g = R.stack_desc(4, 2048, 8, 256, 512, 4096, 2, [0.9] * 8, pos=10)
    need = R.lib.retnet_decode_workspace_size(ctypes.byref(d))
    assert need >= 256 + 4 * (2 * 2048 + 2 * 2048 + 3 * 4096 + 2 * 2048 + 4096)
    dummy = ctypes.c_void_p(256)
    recs = (R.LayerWeights * 2)()
    for i in range(2):
        for k in R.LAYER_KEYS:
            setattr(recs[i], k, 256)
    S = (ctypes.c_void_p * 2)(256, 256)
    # a missing weight, a misaligned state, a small workspace, the third
    # normalisation without z
    recs[1].W2 = None
    assert R.lib.retnet_decode_step(ctypes.byref(d), recs, S, None, dummy, dummy, need, None) == 1
    recs[1].W2 = 256
    S[1] = 260
    assert R.lib.retnet_decode_step(ctypes.byref(d), recs, S, None, dummy, dummy, need, None) == 1
    S[1] = 256
    assert R.lib.retnet_decode_step(ctypes.byref(d), recs, S, None, dummy, dummy, need - 1,
                                    None) == 3
    d4, g4 = R.stack_desc(4, 2048, 8, 256, 512, 4096, 2, [0.9] * 8, pos=10, norm_flags=4)
    need4 = R.lib.retnet_decode_workspace_size(ctypes.byref(d4))
    assert R.lib.retnet_decode_step(ctypes.byref(d4), recs, S, None, dummy, dummy, need4,
                                    None) == 1
    # d_v % 4 != 0 and an empty stack
    d5, g5 = R.stack_desc(4, 64, 2, 16, 6, 32, 1, [0.9] * 2, pos=0)
    assert R.lib.retnet_decode_workspace_size(ctypes.byref(d5)) == 0
    d6, g6 = R.stack_desc(4, 2048, 8, 256, 512, 4096, 0, [0.9] * 8, pos=0)
    assert R.lib.retnet_decode_step(ctypes.byref(d6), None, None, None, None, dummy, 1 << 30,
                                    None) == 0


def test_decode_stack_rejects_overlapping_buffers(R):
    """X and the states are updated in place: a state overlapping X or the
    workspace, or X overlapping the workspace, is refused before any launch
    (only refused calls are made here, so nothing is launched)."""
    d, g = R.stack_desc(4, 2048, 8, 256, 512, 4096, 2, [0.9] * 8, pos=10)
    need = R.lib.retnet_decode_workspace_size(ctypes.byref(d))
    ws = 1 << 32
    X = ws + need + 4096
    recs = (R.LayerWeights * 2)()
    for i in range(2):
        for k in R.LAYER_KEYS:
            setattr(recs[i], k, 1 << 40)
    sbytes = 4 * 8 * 256 * 512 * 4
    base = 1 << 36
    S = (ctypes.c_void_p * 2)(base, base + sbytes)
    call = lambda x, w: R.lib.retnet_decode_step(ctypes.byref(d), recs, S, None,
                                                 ctypes.c_void_p(x), ctypes.c_void_p(w),
                                                 need, None)
    S[1] = X - 256          # state ends inside X
    assert call(X, ws) == 1
    S[1] = ws + need - 1024  # state starts inside the workspace
    assert call(X, ws) == 1
    S[1] = base + sbytes
    assert call(ws + 512, ws) == 1  # X inside the workspace


def test_binding_rejects_host_tensors(R):
    """A tensor that is not on the current CUDA device never reaches a kernel:
    the binding raises before the library is called."""
    import torch
    from linear_recurrent_sequence_gb300 import retention
    q = torch.zeros(1, 1, 4, 8, dtype=torch.bfloat16)
    out = torch.empty(1, 1, 4, 8, dtype=torch.bfloat16)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        retention.chunkwise_fwd(q, q, q, [0.9], out=out, workspace=ws)
