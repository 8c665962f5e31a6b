"""The Python binding's marshalling on the host, against a fake library (no GPU).

The binding checks shapes, dtypes, devices and caller-supplied outputs, then
passes data pointers and sizes to the C entry points. Here CPU tensors stand in
for device tensors and a recording fake stands in for libttt_b300.so, so every
check runs and every argument the C call would get can be read back. A wrong
shape, a tensor on another device or a short output must raise before any C
call, since the library sees only pointers and cannot tell.
"""
import ctypes
import contextlib

import pytest
import torch

import test_sequence_layers_06_b300 as ttt


class FakeLib:
    def __init__(self, status=0):
        self.calls = []
        self.status = status

    def __getattr__(self, name):
        if name == "ttt_status_str":
            return lambda s: b"fake status"
        if name in ("ttt_workspace_bytes", "ttt_workspace_bytes_ex", "ttt_linear_bwd_workspace_bytes"):
            return lambda *a: 4096

        def call(*args):
            self.calls.append((name, args))
            return self.status
        return call


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(ttt, "_lib", lib)
    monkeypatch.setattr(ttt, "_is_device_tensor", lambda t: isinstance(t, torch.Tensor))
    monkeypatch.setattr(ttt, "_on_device", lambda device: contextlib.nullcontext())
    monkeypatch.setattr(ttt, "_stream_ptr", lambda stream, device=None: ctypes.c_void_p(0))
    return lib


def linear_args(B=2, H=3, T=40, d=8, dtype=torch.bfloat16):
    Q, K, V = (torch.zeros(B, H, T, d, dtype=dtype) for _ in range(3))
    return Q, K, V, torch.zeros(H), torch.zeros(H, d, d)


def test_linear_forward_marshals_sizes_pointers_and_workspace_bytes(fake):
    Q, K, V, eta, W0 = linear_args()
    ws = torch.zeros(2048, dtype=torch.float32)  # 8 KB, handed over as bytes
    Z, Wo = ttt.ttt_linear_fwd(Q, K, V, eta, W0, 16, workspace=ws)
    (name, a), = fake.calls
    assert name == "ttt_linear_fwd"
    assert [x.value for x in a[:3]] == [Q.data_ptr(), K.data_ptr(), V.data_ptr()]
    assert a[3] == ttt.TTT_BF16 and a[6:11] == (2, 3, 40, 8, 16)
    assert (a[11].value, a[12].value, a[13].value, a[14]) == (Z.data_ptr(), Wo.data_ptr(), ws.data_ptr(), 8192)
    assert Z.shape == Q.shape and Z.dtype == Q.dtype and Wo.shape == (2, 3, 8, 8) and Wo.dtype == torch.float32
    ttt.ttt_linear_fwd(Q, K, V, eta, W0, 16, options={"force_path": ttt.PATH_SIMT})
    assert fake.calls[-1][0] == "ttt_linear_fwd_ex"


@pytest.mark.parametrize("bad", ["K shape", "V dtype", "eta shape", "W0 dtype", "Z shape", "W_out shape",
                                 "K device", "workspace device", "K strided"])
def test_linear_forward_refuses_before_the_call(fake, bad):
    Q, K, V, eta, W0 = linear_args()
    kw = {}
    if bad == "K shape":
        K = torch.zeros(2, 3, 41, 8, dtype=torch.bfloat16)
    elif bad == "V dtype":
        V = V.float()
    elif bad == "eta shape":
        eta = torch.zeros(4)
    elif bad == "W0 dtype":
        W0 = W0.double()
    elif bad == "Z shape":
        kw["Z"] = torch.zeros(2, 3, 39, 8, dtype=torch.bfloat16)
    elif bad == "W_out shape":
        kw["W_out"] = torch.zeros(2, 3, 8, 7)
    elif bad == "K device":
        K = torch.zeros(2, 3, 40, 8, dtype=torch.bfloat16, device="meta")
    elif bad == "workspace device":
        kw["workspace"] = torch.zeros(4096, dtype=torch.uint8, device="meta")
    elif bad == "K strided":
        K = torch.zeros(2, 3, 8, 40, dtype=torch.bfloat16).transpose(2, 3)
    with pytest.raises((TypeError, ValueError)):
        ttt.ttt_linear_fwd(Q, K, V, eta, W0, 16, **kw)
    assert fake.calls == []


def test_mlp_checks_caller_outputs(fake):
    B, H, T, d = 1, 2, 32, 8
    Q, K, V = (torch.zeros(B, H, T, d, dtype=torch.bfloat16) for _ in range(3))
    eta, W1, W2 = torch.zeros(H), torch.zeros(H, d, 4 * d), torch.zeros(H, 4 * d, d)
    for fn in (ttt.ttt_mlp_fwd, ttt.ttt_mlp_fwd_noalloc):
        for kw in ({"Z": torch.zeros(B, H, T - 1, d, dtype=torch.bfloat16)}, {"W1_out": torch.zeros(B, H, d, d)},
                   {"W2_out": torch.zeros(B, H, 4 * d, d, dtype=torch.bfloat16)}):
            with pytest.raises((TypeError, ValueError)):
                fn(Q, K, V, eta, W1, W2, 16, **kw)
    assert fake.calls == []
    Z, A1, A2 = ttt.ttt_mlp_fwd(Q, K, V, eta, W1, W2, 16)
    Z, A1, A2 = ttt.ttt_mlp_fwd_noalloc(Q, K, V, eta, W1, W2, 16)
    assert [c[0] for c in fake.calls] == ["ttt_mlp_fwd", "ttt_mlp_fwd_noalloc"]
    assert fake.calls[0][1][7:12] == (B, H, T, d, 16) and A1.shape == (B, H, d, 4 * d) and A2.shape == (B, H, 4 * d, d)


def test_decode_checks_its_output_and_states(fake):
    B, H, d = 2, 3, 8
    q = torch.zeros(B, H, d, dtype=torch.bfloat16)
    eta, Wa, Wr = torch.zeros(H), torch.zeros(B, H, d, d), torch.zeros(B, H, d, d)
    with pytest.raises(ValueError):
        ttt.ttt_linear_decode_step(q, q, q, eta, Wa, Wr, 5, 16, z=torch.zeros(B, H, d - 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        ttt.ttt_linear_decode_step(q, q, q, eta, Wa, torch.zeros(B, H, d, d + 1), 5, 16)
    assert fake.calls == []
    z = ttt.ttt_linear_decode_step(q, q, q, eta, Wa, Wr, 5, 16)
    (name, a), = fake.calls
    assert name == "ttt_linear_decode_step" and a[7:12] == (B, H, d, 5, 16) and a[12].value == z.data_ptr()


def test_backward_marshals_and_refuses_bf16(fake):
    Q, K, V, eta, W0 = linear_args(dtype=torch.float32)
    dZ, dW = torch.zeros_like(Q), torch.zeros(2, 3, 8, 8)
    with pytest.raises(TypeError):
        ttt.ttt_linear_bwd(Q.bfloat16(), K, V, eta, W0, 16, dZ, dW)
    dQ, dK, dV, deta, dW0 = ttt.ttt_linear_bwd(Q, K, V, eta, W0, 16, dZ, dW)
    (name, a), = fake.calls
    assert name == "ttt_linear_bwd" and a[3] == ttt.TTT_F32 and a[6:11] == (2, 3, 40, 8, 16)
    assert a[19] == 4096 and deta.shape == (3,) and dW0.shape == (3, 8, 8) and dQ.shape == Q.shape


def test_a_failed_call_raises_with_its_status(fake):
    fake.status = ttt.TTT_ERR_UNSUPPORTED
    with pytest.raises(ttt.TTTError) as e:
        ttt.ttt_linear_fwd(*linear_args(), 16)
    assert e.value.status == ttt.TTT_ERR_UNSUPPORTED and "fake status" in str(e.value)


def test_stream_must_belong_to_the_tensors_device():
    class Stream:
        def __init__(self, index):
            self.device = torch.device("cuda", index)
            self.cuda_stream = 1234

    assert ttt._stream_ptr(Stream(0), torch.device("cuda", 0)).value == 1234
    with pytest.raises(ValueError):
        ttt._stream_ptr(Stream(1), torch.device("cuda", 0))
