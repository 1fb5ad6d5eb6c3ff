"""Helpers for the GPU parity tests: read the library's workspace back into the
oracle's logical layouts, and compare outputs with the stated tolerances."""
import numpy as np
import torch


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def read_workspace(ws, mode: int) -> dict:
    """Device workspace -> numpy arrays in the oracle's logical (unpadded) layouts."""
    s, L = ws.shape, ws.layout
    B, Hq, Hkv, N, M, d = s.B, s.Hq, s.Hkv, s.N, s.M, s.d
    Np, Mp, Tm, Tn = L.N_pad, L.M_pad, L.Tm, L.Tn
    cb = 2 if mode in (0, 3) else 1  # INT8 codes (modes 0 and 3) are held as fp16 values

    def f32(name, n):
        return _np(ws.region(name, 4 * n).view(torch.float32))

    qraw = ws.region("qhat", B * Hq * Np * d * cb)
    kraw = ws.region("khat", B * Hkv * Mp * d * cb)
    if mode in (0, 3):
        qc = _np(qraw.view(torch.float16)).astype(np.float32).reshape(B, Hq, Np, d)[:, :, :N]
        kc = _np(kraw.view(torch.float16)).astype(np.float32).reshape(B, Hkv, Mp, d)[:, :, :M]
        assert np.all(qc == np.round(qc)) and np.all(np.abs(qc) <= 127)
        qc = qc.astype(np.int8).view(np.uint8)
        kc = kc.astype(np.int8).view(np.uint8)
    else:
        qc = _np(qraw).reshape(B, Hq, Np, d)[:, :, :N]
        kc = _np(kraw).reshape(B, Hkv, Mp, d)[:, :, :M]
    if mode == 3:  # SageBwd: per-block INT8 V as fp16 values
        vf = _np(ws.region("vhat", B * Hkv * d * Mp * 2).view(torch.float16)).astype(np.float32)
        vf = vf.reshape(B, Hkv, d, Mp)
        assert np.all(vf == np.round(vf)) and np.all(np.abs(vf) <= 127)
        vt = vf[..., :M].astype(np.int8).view(np.uint8)
        pad_v = vf[..., M:]
    else:
        vt = _np(ws.region("vhat", B * Hkv * d * Mp)).reshape(B, Hkv, d, Mp)[..., :M]
        pad_v = vt_pad(ws, B, Hkv, d, Mp, M)
    extra = {}
    if mode == 3:
        extra["dvb"] = f32("dvb", B * Hkv * Tn).reshape(B, Hkv, Tn)
    return dict(extra,
        qc=np.ascontiguousarray(qc), kc=np.ascontiguousarray(kc),
        vc=np.ascontiguousarray(vt.transpose(0, 1, 3, 2)),
        dq=f32("dq", B * Hq * Tm).reshape(B, Hq, Tm),
        qbar=f32("qbar", B * Hq * Tm * d).reshape(B, Hq, Tm, d),
        dk=f32("dk", B * Hkv * Tn).reshape(B, Hkv, Tn),
        kbar=f32("kbar", B * Hkv * d).reshape(B, Hkv, d),
        dv=f32("dv", B * Hkv * d).reshape(B, Hkv, d),
        vm=f32("vm", B * Hkv * d).reshape(B, Hkv, d),
        dqt=f32("dqt", B * Hq * Np).reshape(B, Hq, Np)[:, :, :N],
        pad_q=_np(qraw).reshape(B, Hq, Np, d * cb)[:, :, N:],
        pad_v=pad_v,
    )


def _nibbles(b: np.ndarray) -> np.ndarray:
    """packed bytes [..., n] -> E2M1 codes [..., 2n] (element 2i in the low nibble)"""
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def _atom_scales(atoms: np.ndarray, rows: int, groups: int) -> np.ndarray:
    """scale atoms [tiles, groups/4, 512] -> scales [tiles*128 rows, groups]:
    row r's four block scales of an atom sit at (r % 32) * 16 + (r / 32) * 4"""
    tiles = atoms.shape[0]
    r = np.arange(128)
    out = np.empty((tiles, 128, groups), np.uint8)
    for g in range(groups):
        out[:, :, g] = atoms[:, g // 4, (r % 32) * 16 + (r // 32) * 4 + (g % 4)]
    return out.reshape(tiles * 128, groups)[:rows]


def read_workspace_fp4(ws) -> dict:
    """NVFP4 workspace -> oracle logical layouts (qc/kc/vc nibbles, qs/ks/vs scales)."""
    s, L = ws.shape, ws.layout
    B, Hq, Hkv, N, M, d = s.B, s.Hq, s.Hkv, s.N, s.M, s.d
    Np, Mp, Tm = L.N_pad, L.M_pad, L.Tm
    G = d // 16
    qc = _nibbles(_np(ws.region("qhat", B * Hq * Np * d // 2)).reshape(B, Hq, Np, d // 2))[:, :, :N]
    kc = _nibbles(_np(ws.region("khat", B * Hkv * Mp * d // 2)).reshape(B, Hkv, Mp, d // 2))[:, :, :M]
    vt = _nibbles(_np(ws.region("vhat", B * Hkv * d * Mp // 2)).reshape(B, Hkv, d, Mp // 2))[..., :M]
    qa = _np(ws.region("qsf", B * Hq * Tm * (d // 64) * 512)).reshape(B * Hq, Tm, d // 64, 512)
    qs = np.stack([_atom_scales(qa[i], N, G) for i in range(B * Hq)]).reshape(B, Hq, N, G)
    ka = _np(ws.region("ksf", B * Hkv * (Mp // 128) * (d // 64) * 512)).reshape(B * Hkv, Mp // 128, d // 64, 512)
    ks = np.stack([_atom_scales(ka[i], M, G) for i in range(B * Hkv)]).reshape(B, Hkv, M, G)
    CA = -(-d // 128)
    va = _np(ws.region("vsf", B * Hkv * CA * (Mp // 64) * 512)).reshape(B * Hkv, CA, Mp // 64, 512)
    Mt16 = -(-M // 16)
    vs = np.empty((B * Hkv, Mt16, d), np.uint8)
    c = np.arange(d)
    for tb in range(Mt16):
        ts, blk = tb // 4, tb % 4
        rr = c % 128
        vs[:, tb, :] = va[:, c // 128, ts, (rr % 32) * 16 + (rr // 32) * 4 + blk]
    f32 = lambda name, n: _np(ws.region(name, 4 * n).view(torch.float32))
    return dict(qc=np.ascontiguousarray(qc), kc=np.ascontiguousarray(kc),
                vc=np.ascontiguousarray(vt.transpose(0, 1, 3, 2)), qs=qs, ks=ks,
                vs=vs.reshape(B, Hkv, Mt16, d),
                qbar=f32("qbar", B * Hq * Tm * d).reshape(B, Hq, Tm, d),
                kbar=f32("kbar", B * Hkv * d).reshape(B, Hkv, d),
                vm=f32("vm", B * Hkv * d).reshape(B, Hkv, d))


def compare_codes_fp4(got: dict, ref) -> dict:
    def fold(c):  # -0 (0x8) and +0 both encode zero
        c = c.copy()
        c[c == 0x8] = 0
        return c

    def bits(a):
        return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)

    return dict(qc=np.array_equal(fold(got["qc"]), fold(ref.qc)), kc=np.array_equal(fold(got["kc"]), fold(ref.kc)),
                vc=np.array_equal(fold(got["vc"]), fold(ref.vc)), qs=np.array_equal(got["qs"], ref.qs),
                ks=np.array_equal(got["ks"], ref.ks), vs=np.array_equal(got["vs"], ref.vs),
                qbar=np.array_equal(bits(got["qbar"]), bits(ref.qbar)),
                kbar=np.array_equal(bits(got["kbar"]), bits(ref.kbar)),
                vm=np.array_equal(bits(got["vm"]), bits(ref.vm)))


def vt_pad(ws, B, Hkv, d, Mp, M):
    vt = _np(ws.region("vhat", B * Hkv * d * Mp)).reshape(B, Hkv, d, Mp)
    return vt[..., M:]


def fold_neg_zero_e4m3(c: np.ndarray) -> np.ndarray:
    """E4M3 codes with -0 (0x80) folded onto +0: both encode zero."""
    c = c.copy()
    c[c == 0x80] = 0
    return c


def compare_codes(got: dict, ref, mode: int, flags: int):
    """Bit-exact comparison of codes, scales and means (E4M3 +-0 folded)."""
    def bits(a):
        return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)

    qc_ref, kc_ref, vc_ref = ref.qc, ref.kc, ref.vc
    qc, kc, vc = got["qc"], got["kc"], got["vc"]
    if mode == 1:
        qc, kc, qc_ref, kc_ref = map(fold_neg_zero_e4m3, (qc, kc, qc_ref, kc_ref))
    if mode != 3:  # E4M3 V codes
        vc, vc_ref = fold_neg_zero_e4m3(vc), fold_neg_zero_e4m3(vc_ref)
    out = {}
    out["dq"] = np.array_equal(bits(got["dq"]), bits(ref.dq))
    out["dk"] = np.array_equal(bits(got["dk"]), bits(ref.dk))
    if mode == 3:  # per-block V scales (the per-channel ones are not part of this mode)
        out["dvb"] = np.array_equal(bits(got["dvb"]), bits(ref.dvb))
    else:
        out["dv"] = np.array_equal(bits(got["dv"]), bits(ref.dv))
    out["kbar"] = np.array_equal(bits(got["kbar"]), bits(ref.kbar))
    out["vm"] = np.array_equal(bits(got["vm"]), bits(ref.vm))
    out["qbar"] = np.array_equal(bits(got["qbar"]), bits(ref.qbar))
    if flags & 0x10:  # per-token Q scales
        out["dqt"] = np.array_equal(bits(got["dqt"]), bits(ref.dqt))
    out["qc"] = np.array_equal(qc, qc_ref)
    out["kc"] = np.array_equal(kc, kc_ref)
    out["vc"] = np.array_equal(vc, vc_ref)
    out["pad_zero"] = (not got["pad_q"].any()) and (not got["pad_v"].any())
    return out


def output_metrics(got: np.ndarray, ref: np.ndarray) -> dict:
    got = got.astype(np.float64).ravel()
    ref = ref.astype(np.float64).ravel()
    err = np.abs(got - ref)
    return dict(max_rel=float(err.max() / max(np.abs(ref).max(), 1e-30)),
                rel_l1=float(err.sum() / max(np.abs(ref).sum(), 1e-30)),
                cos=float(np.dot(got, ref) / np.sqrt(np.dot(got, got) * np.dot(ref, ref))),
                rmse=float(np.sqrt(np.mean((got - ref) ** 2))))
