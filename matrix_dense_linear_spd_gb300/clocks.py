"""SM clock and clock-event-reason sampling through NVML (ctypes), for the measurement harness.

A background thread reads the SM clock and the active clock-event reasons every few
milliseconds; ``summary(t0, t1)`` gives the median SM clock and the reasons seen inside a
wall-clock window, so a timing can be checked for throttling or a clock lock. Read-only: no
GPU setting is changed.
"""
from __future__ import annotations

import ctypes
import statistics
import threading
import time


class ClockSampler:
    """Samples SM clock and clock-event reasons every few ms in a background thread."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device: int = 0, period: float = 0.005):
        self.period = period
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            import torch
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(torch_device).uuid)
            except Exception:
                pass
            rc = 1
            if uuid:
                for cand in (uuid, "GPU-" + uuid):
                    rc = self.nvml.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(self.handle))
                    if rc == 0:
                        break
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.handle))
            if rc != 0:
                raise OSError("no NVML handle")
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except Exception:
            self.ok = False

    def _one(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(c)) != 0:
            return
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(r))
        self.samples.append((time.perf_counter(), c.value, r.value))

    def _run(self):
        while not self._stop.is_set():
            self._one()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self, t0=None, t1=None):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable"}
        sel = [s for s in self.samples if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        if len(sel) < 3:
            sel = self.samples
        reasons = set()
        for _, _, r in sel:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sel), "source": "nvml"}
